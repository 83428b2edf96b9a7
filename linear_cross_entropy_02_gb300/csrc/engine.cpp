// Host engine behind the C ABI of include/flce.h: argument checks, workspace
// carving, tensor-map encoding, and the stream-ordered launch sequence of the
// row-chunk loop. No allocation, no host synchronisation (except in
// flce_get_status and flce_profile_read, which exist to synchronise).
//
// Launch sequence of flce_forward_backward (one stream):
//   prologue                               labels -> n_valid, status, sums = 0
//   [W^T transpose]                        when grad_h is wanted
//   for each chunk of C rows:
//     forward GEMM + statistics epilogue   z = m h_c W^T, s = cap(z) stored (fp16
//                                          s - gmax per 32 columns on the bf16 path)
//     merge                                lse, argmax, row loss, chunk sums
//     dlogits                              dz (bf16); dz^T on the K-major paths
//     grad_h GEMM                          grad_h_c = m dz W
//     [h_c^T transpose] + grad_W GEMM      grad_W += m dz^T h_c
//   finish                                 loss, token accuracy
// The logits of a chunk are the only O(C * V) transient (the Liger-Kernel
// DeepSeek-V3 page, section Memory: chunked transients instead of the full
// logits). FLCE_FLAG_RECOMPUTE and the vocabulary-parallel backward keep none:
// they rebuild the logits per vocab slab (recompute_slabs).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>
#include <vector>

#include "flce_internal.h"

using namespace flce;

namespace {

constexpr int64_t kDefaultChunkRows = 8192;
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;
constexpr int kMaxDevices = 64;

std::atomic<int64_t> g_launches{0};

// ------------------------------------------------------------ profiling
struct ProfRecord {
  int kernel;
  cudaEvent_t start, stop;
};
std::mutex g_prof_mu;
bool g_prof_on = false;
std::vector<ProfRecord> g_prof;

struct LaunchScope {
  int kernel;
  cudaStream_t stream;
  cudaEvent_t start = nullptr, stop = nullptr;
  LaunchScope(int k, cudaStream_t s) : kernel(k), stream(s) {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    if (!g_prof_on) return;
    if (cudaEventCreate(&start) != cudaSuccess) {
      start = nullptr;
    } else if (cudaEventCreate(&stop) != cudaSuccess) {
      cudaEventDestroy(start);
      start = stop = nullptr;
    } else {
      cudaEventRecord(start, stream);
    }
  }
  ~LaunchScope() {
    g_launches.fetch_add(1);
    if (start) {
      cudaEventRecord(stop, stream);
      std::lock_guard<std::mutex> lk(g_prof_mu);
      g_prof.push_back({kernel, start, stop});
    }
  }
};

const char* const kKernelNames[FLCE_NUM_KERNELS] = {
    "prologue", "fwd_gemm_stats", "merge", "dlogits", "grad_h_gemm",
    "grad_W_gemm", "transpose_W", "transpose_h", "finish", "simt_stats",
    "ce_stats", "ce_grad", "recompute_dz_gemm", "convert_grad_h", "scale_gradient", "vp_merge",
    "split_tf32"};

// ------------------------------------------------------------ device info
// Per-device cache of the SM count and compute capability, packed into one
// atomic word (cc << 16 | sms; 0 = not yet queried) so that host threads
// making their first calls at once neither race nor see half an entry.
std::atomic<uint32_t> g_dev_info[kMaxDevices] = {};

int device_info(int* sms, int* cc) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FLCE_ERR_CUDA;
  uint32_t v = g_dev_info[dev].load(std::memory_order_acquire);
  if (v == 0) {
    int n = 0, major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return FLCE_ERR_CUDA;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return FLCE_ERR_CUDA;
    if (cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) return FLCE_ERR_CUDA;
    v = (static_cast<uint32_t>(major * 10 + minor) << 16) | (static_cast<uint32_t>(n) & 0xffffu);
    g_dev_info[dev].store(v, std::memory_order_release);
  }
  *sms = static_cast<int>(v & 0xffffu);
  *cc = static_cast<int>(v >> 16);
  return FLCE_OK;
}

// ------------------------------------------------------------ tensor maps
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool load_encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
  });
  return g_encode != nullptr;
}

// bf16 [outer][inner] with row stride `ld` elements; box = 64 x box_rows, 128-byte swizzle.
bool encode_bf16(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t ld, uint32_t box_rows) {
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {ld * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// fp32 operand [outer][inner] with row stride `ld` elements, read as tf32:
// box = 32 x box_rows (one 128-byte swizzle row per operand row).
bool encode_f32_in(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t ld,
                   uint32_t box_rows) {
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {ld * 4};
  cuuint32_t box[2] = {32, box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// fp32 [outer][inner] with row stride `ld` elements; 32 x 32 boxes (128-byte
// rows), 128-byte swizzle: the epilogue's bulk store / reduce-add target.
bool encode_f32_out(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t ld) {
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {ld * 4};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t es[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// fp16 [outer][inner] with row stride `ld` elements; 64 x 32 boxes (128-byte
// rows), 128-byte swizzle: the forward epilogue's store of s - gmax.
bool encode_f16_out(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t ld) {
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {ld * 2};
  cuuint32_t box[2] = {64, 32};
  cuuint32_t es[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// ------------------------------------------------------------ layout
inline int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

struct Layout {
  int64_t C;        // rows per chunk (multiple of 128)
  int64_t n_vtiles; // vocab tiles of 256
  int64_t ldp, ldz, ldd, ldt, ldwt, ldht;
  int64_t merge_blocks;
  int64_t slab;     // recompute mode: vocab columns per slab (0 otherwise)
  bool need_z, need_dz, need_dzt, need_wt, need_ht, need_gh32;
  // z16: the stored logits are fp16 s - gmax with fp32 gmax per 32 columns
  // (the bf16 backward on MN-major tiles); otherwise fp32 s
  bool z16;
  int64_t ldg;      // gmax row stride (ldz / 32)
  size_t off_hdr, off_bl, off_bc, off_pmax, off_psum, off_pidx, off_tgt, off_lse, off_z, off_gmax, off_dz, off_dzt,
      off_wt, off_ht, off_gh32, total;
  // three-pass tf32 (fp32 operands with FLCE_FLAG_F32_3PASS): hi / lo copies
  // of W and h_c for the forward GEMM, and lo halves beside W^T, h_c^T, dz
  // and dz^T (which then hold the hi halves)
  bool split;
  size_t off_whi, off_wlo, off_hhi, off_hlo, off_wtlo, off_htlo, off_dzlo, off_dztlo;
  // host inputs (flce_forward_backward_from_host): two chunk buffers of h, all
  // labels, and the two result scalars before they are copied to the host
  bool host_in;
  size_t off_hstage, hstage_bytes, off_labels, off_out;
};

struct Norm {
  flce_params p;
  int64_t ld_h, ld_w;
};

// need_hidden = false for the cross-entropy on materialised logits, which has
// no hidden dimension (p->hidden, ld_h, ld_w are ignored there).
int normalise(const flce_params* in, Norm* out, bool need_hidden = true) {
  if (!in) return FLCE_ERR_ARG;
  Norm n;
  n.p = *in;
  if (!need_hidden) {
    n.p.hidden = 8;
    n.p.ld_h = n.p.ld_w = 0;
  }
  const flce_params& p = n.p;
  if (p.n_rows < 0 || p.hidden <= 0 || p.vocab <= 0 || p.vocab >= (int64_t(1) << 31) - 512) return FLCE_ERR_ARG;
  if (p.n_rows >= (int64_t(1) << 31) - 512 || p.hidden >= (int64_t(1) << 24)) return FLCE_ERR_ARG;
  if (!(p.softcap >= 0.f) || !std::isfinite(p.softcap) || !std::isfinite(p.out_mult) ||
      !std::isfinite(p.grad_scale))
    return FLCE_ERR_ARG;
  if (p.reduction != FLCE_REDUCTION_MEAN && p.reduction != FLCE_REDUCTION_SUM &&
      !(p.reduction == FLCE_REDUCTION_NONE && !need_hidden))
    return FLCE_ERR_ARG;
  if (p.chunk_rows < 0 || p.timeout_ns < 0) return FLCE_ERR_ARG;
  if (p.dtype != FLCE_DTYPE_BF16 && p.dtype != FLCE_DTYPE_F32) return FLCE_ERR_ARG;
  if (p.hidden % 8 != 0) return FLCE_ERR_ALIGN;
  n.ld_h = p.ld_h == 0 ? p.hidden : p.ld_h;
  n.ld_w = p.ld_w == 0 ? p.hidden : p.ld_w;
  if (n.ld_h < p.hidden || n.ld_w < p.hidden) return FLCE_ERR_ARG;
  if (n.ld_h % 8 != 0 || n.ld_w % 8 != 0) return FLCE_ERR_ALIGN;
  *out = n;
  return FLCE_OK;
}

// ------------------------------------------------------------ default chunk
// Predicted cost of one tcgen05 GEMM in units of one 128-row tile's K step:
// the waves of its persistent grid in 128 x 256 tiles, or 1.82 per wave of
// 256 x 256 tiles where those finish first (the rule pick_wide applies at
// launch), times its K steps.
constexpr int kTunedSms = 152;  // GB300

double gemm_cost(int64_t m_tiles, int64_t n_tiles, int64_t k_iters, int flags) {
  const int64_t narrow = (m_tiles * n_tiles + kTunedSms - 1) / kTunedSms;
  const int64_t wide = (((m_tiles + 1) / 2) * n_tiles + kTunedSms - 1) / kTunedSms;
  double waves = std::min<double>(static_cast<double>(narrow), 1.82 * static_cast<double>(wide));
  if (flags & FLCE_FLAG_TILE128) waves = static_cast<double>(narrow);
  if (flags & FLCE_FLAG_TILE256) waves = 1.82 * static_cast<double>(wide);
  return waves * static_cast<double>(k_iters);
}

// The forward, grad_h and grad_W GEMMs of one chunk of `rows` rows.
double chunk_cost(int64_t rows, int64_t H, int64_t V, bool gh, bool gw, int flags) {
  const int64_t m = (rows + kBM - 1) / kBM;
  double t = gemm_cost(m, (V + kBN - 1) / kBN, (H + kBK - 1) / kBK, flags);
  if (gh) t += gemm_cost(m, (H + kBN - 1) / kBN, (V + kBK - 1) / kBK, flags);
  if (gw) t += gemm_cost((V + kBM - 1) / kBM, (H + kBN - 1) / kBN, (rows + kBK - 1) / kBK, flags);
  return t;
}

// Rows per chunk when the caller leaves chunk_rows at 0, for the stored-logits
// backward: among multiples of 256 from 8192 to 10240, the one whose chunks
// (the last one ragged) give the lowest predicted GEMM cost; 8192 on ties.
// It matters where a GEMM's tile count leaves its last wave nearly empty: on
// the frozen 131072 x 4096 x 151936 head, grad_h on 8192-row chunks takes 7
// waves of 128-row tiles per chunk, on 9728-row chunks exactly 4 waves of
// 256-row tiles, and the forward + grad_h step went from 212.0 to 202.4 ms.
// The other calls keep 8192 rows.
int64_t default_chunk_rows(int64_t N, int64_t H, int64_t V, bool gh, bool gw, int flags) {
  auto total = [&](int64_t C) {
    const int64_t full = N / C, rem = N % C;
    return static_cast<double>(full) * chunk_cost(C, H, V, gh, gw, flags) +
           (rem > 0 ? chunk_cost(rem, H, V, gh, gw, flags) : 0.0);
  };
  int64_t best = kDefaultChunkRows;
  double best_t = total(best);
  for (int64_t C = kDefaultChunkRows + 256; C <= 10240; C += 256) {
    const double t = total(C);
    if (t < best_t * (1.0 - 1e-9)) {
      best = C;
      best_t = t;
    }
  }
  return best;
}

// z_rows: rows of the stored-logit region (0: one chunk, C; the kept logits of
// FLCE_FLAG_VP_STORED hold all N rows).
void make_layout(const Norm& n, int mode, bool gh, bool gw, Layout* L, int64_t z_rows = 0) {
  const flce_params& p = n.p;
  L->host_in = mode == FLCE_MODE_FORWARD_BACKWARD_HOST || mode == FLCE_MODE_CE_ONLY_HOST;
  if (mode == FLCE_MODE_FORWARD_BACKWARD_HOST) mode = FLCE_MODE_FORWARD_BACKWARD;
  if (mode == FLCE_MODE_CE_ONLY_HOST) mode = FLCE_MODE_CE_ONLY;
  const bool ce = mode == FLCE_MODE_CROSS_ENTROPY;
  const bool simt = !ce && (p.flags & FLCE_FLAG_SIMT_GEMM) != 0;
  const bool bwd = mode == FLCE_MODE_FORWARD_BACKWARD && (gh || gw);
  const bool tuned = bwd && !simt && p.dtype == FLCE_DTYPE_BF16 &&
                     (p.flags & (FLCE_FLAG_RECOMPUTE | FLCE_FLAG_KMAJOR_BWD)) == 0 && p.n_rows > kDefaultChunkRows;
  int64_t c = p.chunk_rows > 0 ? p.chunk_rows
              : tuned        ? default_chunk_rows(p.n_rows, p.hidden, p.vocab, gh, gw, p.flags)
                             : kDefaultChunkRows;
  c = std::min<int64_t>(c, std::max<int64_t>(p.n_rows, 1));
  c = std::min<int64_t>(c, 32768);  // grid.y of the row-streaming kernels stays below 65536
  L->C = round_up(c, kBM);
  L->n_vtiles = ce ? (p.vocab + kCeTile - 1) / kCeTile : (p.vocab + kVTile - 1) / kVTile;
  L->ldp = L->C;
  L->ldz = L->n_vtiles * kVTile;
  L->ldd = round_up(p.vocab, 8);
  L->ldt = L->C;
  L->ldwt = round_up(p.vocab, 8);
  L->ldht = L->C;
  L->merge_blocks = (L->C + kMergeRows - 1) / kMergeRows;
  // The backward GEMMs read W, dz and h_c in place as MN-major tiles; the
  // transposed copies exist only on the debug paths (SIMT GEMMs, or the
  // K-major cross-check flag).
  // The recompute mode keeps no logits: a [C][slab] bf16 dlogits slab and an
  // fp32 [C][H] grad_h accumulator instead.
  // fp32 operands (tf32 GEMMs) take the all-K-major backward with fp32 dz and
  // fp32 transposed copies; the recompute mode is bf16 only.
  const bool f32 = p.dtype == FLCE_DTYPE_F32;
  const bool recompute = bwd && !simt && !f32 && (p.flags & FLCE_FLAG_RECOMPUTE) != 0;
  const bool kmajor = !recompute && (simt || f32 || (p.flags & FLCE_FLAG_KMAJOR_BWD) != 0);
  const size_t es = f32 ? 4 : 2;  // element size of dz, dz^T, W^T, h_c^T
  L->slab = 0;
  if (recompute) {
    const int64_t want = p.vocab_slab > 0 ? p.vocab_slab : 16384;
    L->slab = round_up(std::min<int64_t>(want, round_up(p.vocab, kVTile)), kVTile);
  }
  L->need_z = (bwd && !recompute) || simt;
  L->z16 = bwd && !recompute && !simt && !kmajor && !f32;
  L->ldg = L->ldz / 32;
  L->need_dz = bwd && (gh || (gw && !kmajor));
  L->need_dzt = bwd && gw && kmajor;
  L->need_wt = bwd && gh && kmajor;
  L->need_ht = bwd && gw && kmajor;
  L->need_gh32 = recompute && gh;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += (bytes + 255) / 256 * 256;
    return o;
  };
  L->off_hdr = take(sizeof(Header));
  L->off_bl = take(sizeof(double) * L->merge_blocks);
  L->off_bc = take(sizeof(int64_t) * L->merge_blocks);
  L->off_pmax = take(sizeof(float) * L->n_vtiles * L->ldp);
  L->off_psum = take(sizeof(float) * L->n_vtiles * L->ldp);
  L->off_pidx = take(sizeof(int32_t) * L->n_vtiles * L->ldp);
  L->off_tgt = take(sizeof(float) * L->C);
  L->off_lse = take(sizeof(float) * L->C);
  const int64_t zr = z_rows > 0 ? z_rows : L->C;
  L->off_z = L->need_z ? take((L->z16 ? 2 : sizeof(float)) * zr * L->ldz) : 0;
  L->off_gmax = L->z16 ? take(sizeof(float) * zr * L->ldg) : 0;
  L->off_dz = L->need_dz ? take(es * L->C * (recompute ? L->slab : L->ldd)) : 0;
  L->off_dzt = L->need_dzt ? take(es * round_up(p.vocab, kBM) * L->ldt) : 0;
  L->off_wt = L->need_wt ? take(es * p.hidden * L->ldwt) : 0;
  L->off_ht = L->need_ht ? take(es * p.hidden * L->ldht) : 0;
  L->off_gh32 = L->need_gh32 ? take(sizeof(float) * L->C * p.hidden) : 0;
  L->split = f32 && !ce && (p.flags & FLCE_FLAG_F32_3PASS) != 0;
  L->off_whi = L->split ? take(sizeof(float) * p.vocab * p.hidden) : 0;
  L->off_wlo = L->split ? take(sizeof(float) * p.vocab * p.hidden) : 0;
  L->off_hhi = L->split ? take(sizeof(float) * L->C * p.hidden) : 0;
  L->off_hlo = L->split ? take(sizeof(float) * L->C * p.hidden) : 0;
  L->off_wtlo = L->split && L->need_wt ? take(es * p.hidden * L->ldwt) : 0;
  L->off_htlo = L->split && L->need_ht ? take(es * p.hidden * L->ldht) : 0;
  L->off_dzlo = L->split && L->need_dz ? take(es * L->C * L->ldd) : 0;
  L->off_dztlo = L->split && L->need_dzt ? take(es * round_up(p.vocab, kBM) * L->ldt) : 0;
  const size_t h_es = p.dtype == FLCE_DTYPE_F32 ? 4 : 2;
  L->hstage_bytes = L->host_in ? (static_cast<size_t>(L->C) * p.hidden * h_es + 255) / 256 * 256 : 0;
  L->off_hstage = L->host_in ? take(2 * L->hstage_bytes) : 0;
  L->off_labels = L->host_in ? take(sizeof(int64_t) * std::max<int64_t>(p.n_rows, 1)) : 0;
  L->off_out = L->host_in ? take(2 * sizeof(float)) : 0;
  L->total = off;
}

inline bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

// 256-row CTA tiles carry a third less operand traffic into each SM per flop
// than 128-row tiles, which the tensor cores otherwise wait on: a 256-row tile
// costs about 1.82 128-row tiles (measured on the DSV3 head). With few tiles
// the coarser grid can lose more to the last partial wave than that saves, so
// each GEMM takes the shape with the shorter makespan of the persistent grid,
// unless a flag fixes it.
bool pick_wide(int flags, const GemmParams& g, int sms) {
  if (flags & FLCE_FLAG_TILE128) return false;
  if (flags & FLCE_FLAG_TILE256) return true;
  const int64_t narrow = (static_cast<int64_t>(g.m_tiles) * g.n_tiles + sms - 1) / sms;
  const int64_t units = static_cast<int64_t>((g.m_tiles + 1) / 2) * g.n_tiles;
  const int64_t wide_waves = (units + sms - 1) / sms;
  return 182 * wide_waves < 100 * narrow;
}

#define FLCE_LAUNCH(kid, expr)                         \
  do {                                                 \
    LaunchScope _scope((kid), stream);                 \
    if ((expr) != cudaSuccess) return FLCE_ERR_CUDA;   \
  } while (0)

struct Call {
  int mode;  // FLCE_MODE_*; host inputs come as FORWARD_BACKWARD or CE_ONLY with host_in set
  const void* h;
  const void* W;
  const int64_t* labels;
  float* loss;
  float* acc;
  int64_t* predicted;
  float* row_lse;
  void* grad_h;
  float* grad_W;
  void* ws;
  size_t ws_bytes;
  cudaStream_t stream;
  // host inputs: h and labels are host pointers, staged chunk by chunk on
  // copy_stream; loss / acc are then host pointers written at the end
  bool host_in = false;
  cudaStream_t copy_stream = nullptr;
  // vocab shard (flce_vp_forward): W holds vocab ids [vocab_offset,
  // vocab_offset + p->vocab) of vocab_total; the per-row partials go to
  // shard_partials ([4][N]) instead of the loss and predictions
  int64_t vocab_offset = 0;
  int64_t vocab_total = 0;
  float* shard_partials = nullptr;
  bool shard_call = false;
  // FLCE_FLAG_VP_STORED: the shard forward stores its logits in the layout
  // that the shard backward will read them from (make_vp_stored_layout)
  bool vp_stored = false;
};

int run_f32(const Norm& n, const Call& c);
// Chunked host-to-device staging of h for host inputs. Chunk k (rows
// [kC, kC + C)) is copied on the copy stream into buffer k % 2 of the
// workspace: `copied[b]` tells the compute stream it has landed, `freed[b]`
// tells the copy stream that every kernel of the chunk that used the buffer
// before has been enqueued ahead of it, so the copy may overwrite it.
struct HostStaging {
  uint8_t* buf[2] = {nullptr, nullptr};
  const uint8_t* src = nullptr;
  size_t ld_bytes = 0, row_bytes = 0;
  int64_t n_rows = 0, C = 0;
  cudaStream_t compute = nullptr, copy = nullptr;
  cudaEvent_t copied[2] = {nullptr, nullptr}, freed[2] = {nullptr, nullptr};

  bool init(uint8_t* base, size_t buf_bytes, const void* h_host, int64_t ld_h, int64_t H, size_t elem_bytes,
            int64_t rows, int64_t chunk, cudaStream_t comp, cudaStream_t cp) {
    buf[0] = base;
    buf[1] = base + buf_bytes;
    src = static_cast<const uint8_t*>(h_host);
    ld_bytes = static_cast<size_t>(ld_h) * elem_bytes;
    row_bytes = static_cast<size_t>(H) * elem_bytes;
    n_rows = rows;
    C = chunk;
    compute = comp;
    copy = cp;
    for (int b = 0; b < 2; ++b) {
      if (cudaEventCreateWithFlags(&copied[b], cudaEventDisableTiming) != cudaSuccess) return false;
      if (cudaEventCreateWithFlags(&freed[b], cudaEventDisableTiming) != cudaSuccess) return false;
    }
    // The first copies wait for everything already on the compute stream: an
    // earlier call on the same workspace may still be reading the buffers.
    if (cudaEventRecord(freed[0], compute) != cudaSuccess) return false;
    if (cudaStreamWaitEvent(copy, freed[0], 0) != cudaSuccess) return false;
    return issue(0) && issue(1);
  }
  bool issue(int64_t k) {
    const int64_t r0 = k * C;
    if (r0 >= n_rows) return true;
    const int64_t rows = std::min<int64_t>(C, n_rows - r0);
    const int b = static_cast<int>(k & 1);
    if (k >= 2 && cudaStreamWaitEvent(copy, freed[b], 0) != cudaSuccess) return false;
    if (cudaMemcpy2DAsync(buf[b], row_bytes, src + r0 * ld_bytes, ld_bytes, row_bytes, static_cast<size_t>(rows),
                          cudaMemcpyHostToDevice, copy) != cudaSuccess)
      return false;
    return cudaEventRecord(copied[b], copy) == cudaSuccess;
  }
  // Called before chunk k's first kernel: releases chunk k - 1's buffer (all
  // its kernels are enqueued), starts the copy of chunk k + 1 into it, and
  // makes the compute stream wait for chunk k. Returns chunk k's rows.
  const void* wait_chunk(int64_t k) {
    if (k >= 1) {
      if (cudaEventRecord(freed[(k - 1) & 1], compute) != cudaSuccess) return nullptr;
      if (!issue(k + 1)) return nullptr;
    }
    if (cudaStreamWaitEvent(compute, copied[k & 1], 0) != cudaSuccess) return nullptr;
    return buf[k & 1];
  }
  ~HostStaging() {
    for (int b = 0; b < 2; ++b) {  // released once the work recorded on them is done
      if (copied[b]) cudaEventDestroy(copied[b]);
      if (freed[b]) cudaEventDestroy(freed[b]);
    }
  }
};


// Recompute backward of one chunk of rows over vocab slabs (the low-memory
// mode, and each shard of the vocab-parallel backward): per slab of W's rows,
// z is recomputed on the tensor cores and the EPI_DZ epilogue forms bf16
// dlogits from it with the rows' lse; then grad_h += m dz W_slab (fp32
// reduce-add into gh_acc) and grad_W_slab += m dz^T h_c.
// What the backward GEMMs that accumulate in fp32 share: the scale, the
// status word, the wait limit, the tile choice and the stream.
struct AccCtx {
  float alpha;
  Header* hdr;
  uint64_t timeout;
  int flags, sms;
  bool pair;
  cudaStream_t stream;
};

// grad_h part += alpha * dz W over K = V columns: dz [rows][ldd] bf16 (K-major
// A), W [V][ld_w] bf16 read in place (MN-major B); out [rows][H] fp32 gets a
// TMA bulk reduce-add.
int grad_h_acc_gemm(const AccCtx& x, const uint16_t* dz, int64_t ldd, int rows, int V, const uint16_t* W,
                    int64_t ld_w, int H, float* out, int group_m) {
  CUtensorMap map_a, map_b, map_o;
  if (!encode_bf16(&map_a, dz, V, rows, ldd, kBM)) return FLCE_ERR_UNSUPPORTED;
  if (!encode_bf16(&map_b, W, H, V, ld_w, 64)) return FLCE_ERR_UNSUPPORTED;
  if (!encode_f32_out(&map_o, out, H, rows, H)) return FLCE_ERR_UNSUPPORTED;
  GemmParams b{};
  std::memset(&b, 0, sizeof(b));
  b.M = rows;
  b.N = H;
  b.K = V;
  b.m_tiles = (rows + kBM - 1) / kBM;
  b.n_tiles = (H + kBN - 1) / kBN;
  b.k_iters = (V + kBK - 1) / kBK;
  b.group_m = std::min(b.m_tiles, group_m);
  b.alpha = x.alpha;
  b.M_valid = rows;
  b.N_valid = H;
  b.out = out;
  b.ldo = H;
  b.status = &x.hdr->status;
  b.timeout_ns = x.timeout;
  cudaStream_t stream = x.stream;
  FLCE_LAUNCH(K_GRADH_GEMM, launch_gemm_tc(EPI_ACC_F32, false, true, pick_wide(x.flags, b, x.sms), &map_a, &map_b,
                                           &map_o, b, std::min(b.m_tiles * b.n_tiles, x.sms), stream, x.pair));
  return FLCE_OK;
}

// grad_W [V][H] fp32 += alpha * dz^T h_c over K = rows: dz [rows][ldd] and
// h_c [rows][ld_hc] bf16 read in place (both MN-major).
int grad_W_acc_gemm(const AccCtx& x, const uint16_t* dz, int64_t ldd, int rows, int V, const uint16_t* h_c,
                    int64_t ld_hc, int H, float* grad_W) {
  CUtensorMap map_a, map_b, map_o;
  if (!encode_bf16(&map_a, dz, V, rows, ldd, 64)) return FLCE_ERR_UNSUPPORTED;
  if (!encode_bf16(&map_b, h_c, H, rows, ld_hc, 64)) return FLCE_ERR_UNSUPPORTED;
  if (!encode_f32_out(&map_o, grad_W, H, V, H)) return FLCE_ERR_UNSUPPORTED;
  GemmParams b{};
  std::memset(&b, 0, sizeof(b));
  b.M = V;
  b.N = H;
  b.K = rows;
  b.m_tiles = (V + kBM - 1) / kBM;
  b.n_tiles = (H + kBN - 1) / kBN;
  b.k_iters = (rows + kBK - 1) / kBK;
  // Groups of 16 vocab tiles: on the DSV3 head this beat an N-fastest walk
  // with h_c kept in L2 and evict-first dz loads.
  b.group_m = std::min(b.m_tiles, 16);
  b.alpha = x.alpha;
  b.M_valid = V;
  b.N_valid = H;
  b.out = grad_W;
  b.ldo = H;
  b.status = &x.hdr->status;
  b.timeout_ns = x.timeout;
  cudaStream_t stream = x.stream;
  FLCE_LAUNCH(K_GRADW_GEMM, launch_gemm_tc(EPI_ACC_F32, true, true, pick_wide(x.flags, b, x.sms), &map_a, &map_b,
                                           &map_o, b, std::min(b.m_tiles * b.n_tiles, x.sms), stream, x.pair));
  return FLCE_OK;
}

struct SlabArgs {
  int rows, H, V, slab;
  int col_base;              // vocab id of W's row 0 (the shard offset)
  int h_row0;                // row of map_hc holding the chunk's first row
  const CUtensorMap* map_hc; // h (K-major A of the recompute GEMM)
  const CUtensorMap* map_w;  // W (K-major B)
  const CUtensorMap* map_w_pair;  // W with 128-row boxes (CTA-pair tiles), or null
  const uint16_t* h_c;       // the chunk's rows of h, row stride ld_hc
  int64_t ld_hc;
  const uint16_t* W;
  int64_t ld_w;
  const int64_t* labels;     // the chunk's labels
  const float* lse;          // the chunk's lse
  const Header* hdr;
  uint16_t* dz;              // [rows][slab] bf16 workspace
  float* gh_acc;             // [rows][H] fp32, accumulated; null: no grad_h
  float* grad_W;             // [V][H] fp32, accumulated; null: frozen
  const flce_params* p;
  float inv_cap;
  uint64_t timeout;
  int sms;
};

int recompute_slabs(const SlabArgs& a, cudaStream_t stream) {
  const flce_params& p = *a.p;
  Header* hdr = const_cast<Header*>(a.hdr);
  auto wide_for = [&](const GemmParams& g) { return pick_wide(p.flags, g, a.sms); };
  const bool pair = (p.flags & FLCE_FLAG_CTA_PAIR) != 0 && a.map_w_pair != nullptr;
  const int rows = a.rows, H = a.H, V = a.V, slab = a.slab;
  for (int v0 = 0; v0 < V; v0 += slab) {
    const int vs = std::min(slab, V - v0);
    GemmParams r{};
    std::memset(&r, 0, sizeof(r));
    r.M = rows;
    r.N = vs;
    r.K = H;
    r.m_tiles = (rows + kBM - 1) / kBM;
    r.n_tiles = (vs + kBN - 1) / kBN;
    r.k_iters = (H + kBK - 1) / kBK;
    r.group_m = std::min(r.m_tiles, 16);
    r.a_row0 = a.h_row0;
    r.b_row0 = v0;
    r.alpha = p.out_mult;
    r.M_valid = rows;
    r.N_valid = vs;
    r.softcap = p.softcap;
    r.inv_softcap = a.inv_cap;
    r.labels = a.labels;
    r.ignore_index = p.ignore_index;
    r.out = a.dz;
    r.ldo = slab;
    r.lse = a.lse;
    r.hdr = hdr;
    r.grad_scale = p.grad_scale;
    r.reduction = p.reduction;
    r.col0 = a.col_base + v0;
    r.status = &hdr->status;
    r.timeout_ns = a.timeout;
    const bool wr = wide_for(r);
    FLCE_LAUNCH(K_RECOMPUTE_GEMM, launch_gemm_tc(EPI_DZ, false, false, wr, a.map_hc,
                                                 wr && pair ? a.map_w_pair : a.map_w, nullptr, r,
                                                 std::min(r.m_tiles * r.n_tiles, a.sms), stream, pair));
    const AccCtx x{p.out_mult, hdr, a.timeout, p.flags, a.sms, pair, stream};
    // grad_h_c += m dz_slab W_slab, then grad_W_slab += m dz_slab^T h_c
    if (a.gh_acc) {
      const int rc = grad_h_acc_gemm(x, a.dz, slab, rows, vs, a.W + static_cast<int64_t>(v0) * a.ld_w, a.ld_w, H,
                                     a.gh_acc, 8);
      if (rc != FLCE_OK) return rc;
    }
    if (a.grad_W) {
      const int rc = grad_W_acc_gemm(x, a.dz, slab, rows, vs, a.h_c, a.ld_hc, H,
                                     a.grad_W + static_cast<int64_t>(v0) * H);
      if (rc != FLCE_OK) return rc;
    }
  }
  return FLCE_OK;
}

// The workspace layout that FLCE_FLAG_VP_STORED shares between a shard's
// forward and backward: the fused forward + backward layout (chunks of C
// rows) with the fp16 logits and their group maxima kept for all N rows, so
// they and the chunk's dlogits buffer sit at the same offsets in both calls.
void make_vp_stored_layout(const Norm& n, Layout* L) {
  make_layout(n, FLCE_MODE_FORWARD_BACKWARD, true, true, L, std::max<int64_t>(n.p.n_rows, 1));
}

int check_vp_stored(const flce_params& p) {
  if (p.flags & (FLCE_FLAG_RECOMPUTE | FLCE_FLAG_KMAJOR_BWD | FLCE_FLAG_SIMT_GEMM)) return FLCE_ERR_ARG;
  return FLCE_OK;
}

int run(const flce_params* params, const Call& c) {
  Norm n;
  int rc = normalise(params, &n);
  if (rc != FLCE_OK) return rc;
  if (n.p.dtype == FLCE_DTYPE_F32) return run_f32(n, c);
  const flce_params& p = n.p;
  const bool gh = c.mode == FLCE_MODE_FORWARD_BACKWARD && c.grad_h != nullptr;
  const bool gw = c.mode == FLCE_MODE_FORWARD_BACKWARD && c.grad_W != nullptr;
  const bool shard = c.shard_call;
  if ((!c.loss && !shard) || !c.ws || !c.W) return FLCE_ERR_ARG;
  if (p.n_rows > 0 && (!c.h || !c.labels)) return FLCE_ERR_ARG;
  if (!aligned16(c.ws) || (!c.host_in && c.h && !aligned16(c.h)) || !aligned16(c.W)) return FLCE_ERR_ALIGN;
  if (gh && !aligned16(c.grad_h)) return FLCE_ERR_ALIGN;
  if (gw && !aligned16(c.grad_W)) return FLCE_ERR_ALIGN;
  if (c.host_in && (p.flags & (FLCE_FLAG_SIMT_GEMM | FLCE_FLAG_KMAJOR_BWD))) return FLCE_ERR_UNSUPPORTED;
  Layout L;
  make_layout(n, !c.host_in ? c.mode
                             : c.mode == FLCE_MODE_CE_ONLY ? FLCE_MODE_CE_ONLY_HOST : FLCE_MODE_FORWARD_BACKWARD_HOST,
              gh, gw, &L);
  if (c.vp_stored) make_vp_stored_layout(n, &L);  // the logits of all rows are kept for the backward
  if (c.ws_bytes < L.total) return FLCE_ERR_WORKSPACE;
  int sms = 0, cc = 0;
  rc = device_info(&sms, &cc);
  if (rc != FLCE_OK) return rc;
  const bool simt = (p.flags & FLCE_FLAG_SIMT_GEMM) != 0;
  const bool recompute = L.slab > 0;
  const bool kmajor = !recompute && (simt || (p.flags & FLCE_FLAG_KMAJOR_BWD) != 0);
  auto wide_for = [&](const GemmParams& g) { return pick_wide(p.flags, g, sms); };
  if (cc != 103) return FLCE_ERR_UNSUPPORTED;  // the kernels are built for sm_103a only
  if (!simt && !load_encoder()) return FLCE_ERR_UNSUPPORTED;

  cudaStream_t stream = c.stream;
  uint8_t* ws = static_cast<uint8_t*>(c.ws);
  Header* hdr = reinterpret_cast<Header*>(ws + L.off_hdr);
  float* pmax = reinterpret_cast<float*>(ws + L.off_pmax);
  float* psum = reinterpret_cast<float*>(ws + L.off_psum);
  int32_t* pidx = reinterpret_cast<int32_t*>(ws + L.off_pidx);
  float* tgt = reinterpret_cast<float*>(ws + L.off_tgt);
  float* lse = reinterpret_cast<float*>(ws + L.off_lse);
  float* zbuf = L.need_z && !L.z16 ? reinterpret_cast<float*>(ws + L.off_z) : nullptr;
  uint16_t* z16 = L.z16 ? reinterpret_cast<uint16_t*>(ws + L.off_z) : nullptr;
  float* gmax = L.z16 ? reinterpret_cast<float*>(ws + L.off_gmax) : nullptr;
  uint16_t* dz = L.need_dz ? reinterpret_cast<uint16_t*>(ws + L.off_dz) : nullptr;
  uint16_t* dzt = L.need_dzt ? reinterpret_cast<uint16_t*>(ws + L.off_dzt) : nullptr;
  uint16_t* wt = L.need_wt ? reinterpret_cast<uint16_t*>(ws + L.off_wt) : nullptr;
  uint16_t* ht = L.need_ht ? reinterpret_cast<uint16_t*>(ws + L.off_ht) : nullptr;
  const uint64_t timeout = p.timeout_ns > 0 ? static_cast<uint64_t>(p.timeout_ns) : kDefaultTimeoutNs;
  const int N = static_cast<int>(p.n_rows), H = static_cast<int>(p.hidden), V = static_cast<int>(p.vocab);
  const float inv_cap = p.softcap > 0.f ? 1.f / p.softcap : 0.f;

  // Host inputs: the labels go over first (the prologue counts them all);
  // chunk k of h goes to staging buffer k % 2 on copy_stream, at most two
  // chunks ahead of the compute stream, so the copy of chunk k + 1 runs under
  // the GEMMs of chunk k. Events order the two streams both ways.
  const int64_t* labels = c.labels;
  float* out_loss = c.loss;
  float* out_acc = c.acc;
  HostStaging hs;
  if (c.host_in) {
    labels = reinterpret_cast<const int64_t*>(ws + L.off_labels);
    out_loss = reinterpret_cast<float*>(ws + L.off_out);
    out_acc = out_loss + 1;
    if (p.n_rows > 0 &&
        cudaMemcpyAsync(const_cast<int64_t*>(labels), c.labels, sizeof(int64_t) * p.n_rows, cudaMemcpyHostToDevice,
                        stream) != cudaSuccess)
      return FLCE_ERR_CUDA;
    if (!hs.init(ws + L.off_hstage, L.hstage_bytes, c.h, n.ld_h, H, 2, p.n_rows, L.C, stream, c.copy_stream))
      return FLCE_ERR_CUDA;
  }

  const int64_t vocab_total = c.vocab_total > 0 ? c.vocab_total : p.vocab;
  FLCE_LAUNCH(K_PROLOGUE, launch_prologue(labels, p.n_rows, vocab_total, p.ignore_index, hdr, stream));

  CUtensorMap map_h, map_w, map_wt, map_w_pair;
  const bool pair = (p.flags & FLCE_FLAG_CTA_PAIR) != 0 && !simt;
  if (!simt && N > 0) {
    if (!c.host_in && !encode_bf16(&map_h, c.h, H, N, n.ld_h, kBM)) return FLCE_ERR_UNSUPPORTED;
    if (!encode_bf16(&map_w, c.W, H, V, n.ld_w, kBN)) return FLCE_ERR_UNSUPPORTED;
    if (pair && !encode_bf16(&map_w_pair, c.W, H, V, n.ld_w, kBN / 2)) return FLCE_ERR_UNSUPPORTED;
  }
  if (L.need_wt && N > 0) {  // debug paths only
    FLCE_LAUNCH(K_TRANSPOSE_W, launch_transpose_bf16(static_cast<const uint16_t*>(c.W), n.ld_w, V, H, wt, L.ldwt,
                                                     stream));
    if (!simt && !encode_bf16(&map_wt, wt, V, H, L.ldwt, kBN)) return FLCE_ERR_UNSUPPORTED;
  }

  for (int64_t r0 = 0; r0 < p.n_rows; r0 += L.C) {
    const int rows = static_cast<int>(std::min<int64_t>(L.C, p.n_rows - r0));
    const int64_t* lab_c = labels + r0;
    // where this chunk's rows of h are: the caller's array (row r0 of map_h)
    // or the staging buffer the chunk was copied to (row 0 of its own map)
    const uint16_t* h_c = static_cast<const uint16_t*>(c.h) + r0 * n.ld_h;
    int64_t ld_hc = n.ld_h;
    int h_row0 = static_cast<int>(r0);
    CUtensorMap map_hc;
    if (c.host_in) {
      h_c = static_cast<const uint16_t*>(hs.wait_chunk(r0 / L.C));
      if (!h_c) return FLCE_ERR_CUDA;
      ld_hc = H;
      h_row0 = 0;
      if (!encode_bf16(&map_hc, h_c, H, rows, H, kBM)) return FLCE_ERR_UNSUPPORTED;
    } else if (!simt) {
      map_hc = map_h;
    }

    // ---- forward GEMM with the statistics epilogue
    GemmParams g{};
    std::memset(&g, 0, sizeof(g));
    g.M = rows;
    g.N = V;
    g.K = H;
    g.m_tiles = (rows + kBM - 1) / kBM;
    g.n_tiles = static_cast<int>(L.n_vtiles);
    g.k_iters = (H + kBK - 1) / kBK;
    // Groups of 16 row tiles: the group's h_c rows stay in L2 while W streams
    // through once per group. On the DSV3 head, larger groups, and L2
    // evict-last / evict-first policies on either operand, all measured slower:
    // the kept lines crowd the next GEMM's operands out of L2. The stored
    // logits, written once here, do carry evict-first (store_hint): that keeps
    // them from displacing the operands, 1.5-3% on this GEMM.
    g.group_m = std::min(g.m_tiles, 16);
    g.a_row0 = h_row0;
    g.b_row0 = 0;
    g.alpha = p.out_mult;
    g.M_valid = rows;
    g.N_valid = V;
    g.softcap = p.softcap;
    g.inv_softcap = inv_cap;
    g.labels = lab_c;
    g.ignore_index = p.ignore_index;
    g.part_max = pmax;
    g.part_sum = psum;
    g.part_idx = pidx;
    g.tgt = tgt;
    g.ldp = static_cast<int>(L.ldp);
    // kept logits (FLCE_FLAG_VP_STORED): this chunk's rows of the all-row store
    uint16_t* z16_c = z16 && c.vp_stored ? z16 + r0 * L.ldz : z16;
    float* gmax_c = gmax && c.vp_stored ? gmax + r0 * L.ldg : gmax;
    g.zbuf = L.z16 ? nullptr : zbuf;
    g.ldz = L.ldz;
    g.gmax = gmax_c;
    g.ldg = L.ldg;
    g.status = &hdr->status;
    g.timeout_ns = timeout;
    g.debug_flags = p.flags;
    g.col0 = static_cast<int>(c.vocab_offset);
    // without predicted tokens to return, the epilogue keeps only what the
    // token accuracy needs (a shard's partials always carry the argmax)
    g.no_argmax = (c.predicted == nullptr && !shard) ? 1 : 0;
    const bool store = L.need_z;
    g.store_hint = store ? 1 : 0;
    if (simt) {
      FLCE_LAUNCH(K_FWD_GEMM, launch_gemm_simt(EPI_STATS, c.h, n.ld_h, c.W, n.ld_w, g, stream));
      FLCE_LAUNCH(K_SIMT_STATS, launch_stats_from_z(g, rows, store, stream));
    } else {
      const int tiles = g.m_tiles * g.n_tiles;
      CUtensorMap map_z;
      if (store && L.z16 && !encode_f16_out(&map_z, z16_c, L.ldz, rows, L.ldz)) return FLCE_ERR_UNSUPPORTED;
      if (store && !L.z16 && !encode_f32_out(&map_z, zbuf, L.ldz, rows, L.ldz)) return FLCE_ERR_UNSUPPORTED;
      const int mode = !store ? EPI_STATS : L.z16 ? EPI_STATS_STORE16 : EPI_STATS_STORE;
      const bool wg = wide_for(g);
      FLCE_LAUNCH(K_FWD_GEMM, launch_gemm_tc(mode, false, false, wg, &map_hc, wg && pair ? &map_w_pair : &map_w,
                                             store ? &map_z : nullptr, g, std::min(tiles, sms), stream, pair));
    }

    // ---- merge of the vocab-tile statistics
    MergeParams mp{};
    mp.rows = rows;
    mp.n_vtiles = static_cast<int>(L.n_vtiles);
    mp.ldp = static_cast<int>(L.ldp);
    mp.part_max = pmax;
    mp.part_sum = psum;
    mp.part_idx = pidx;
    mp.tgt = tgt;
    mp.labels = lab_c;
    mp.ignore_index = p.ignore_index;
    mp.lse = lse;
    mp.predicted = c.predicted ? c.predicted + r0 : nullptr;
    mp.row_lse = c.row_lse ? c.row_lse + r0 : nullptr;
    mp.block_loss = reinterpret_cast<double*>(ws + L.off_bl);
    mp.block_correct = reinterpret_cast<int64_t*>(ws + L.off_bc);
    mp.hdr = hdr;
    if (shard) {
      mp.shard_out = c.shard_partials + r0;
      mp.ld_shard = p.n_rows;
      mp.vocab_offset = c.vocab_offset;
      mp.vocab_shard = p.vocab;
    }
    FLCE_LAUNCH(K_MERGE, launch_merge(mp, stream));

    if (!gh && !gw) continue;

    if (recompute) {
      // ---- low-memory backward: per vocab slab, recompute z on the tensor
      // cores with dlogits formed in the epilogue, then both backward GEMMs.
      float* gh32 = L.need_gh32 ? reinterpret_cast<float*>(ws + L.off_gh32) : nullptr;
      if (gh32 && cudaMemsetAsync(gh32, 0, sizeof(float) * rows * H, stream) != cudaSuccess) return FLCE_ERR_CUDA;
      SlabArgs sa;
      sa.rows = rows;
      sa.H = H;
      sa.V = V;
      sa.slab = static_cast<int>(L.slab);
      sa.col_base = 0;
      sa.h_row0 = h_row0;
      sa.map_hc = &map_hc;
      sa.map_w = &map_w;
      sa.map_w_pair = pair ? &map_w_pair : nullptr;
      sa.h_c = h_c;
      sa.ld_hc = ld_hc;
      sa.W = static_cast<const uint16_t*>(c.W);
      sa.ld_w = n.ld_w;
      sa.labels = lab_c;
      sa.lse = lse;
      sa.hdr = hdr;
      sa.dz = dz;
      sa.gh_acc = gh32;
      sa.grad_W = gw ? c.grad_W : nullptr;
      sa.p = &p;
      sa.inv_cap = inv_cap;
      sa.timeout = timeout;
      sa.sms = sms;
      rc = recompute_slabs(sa, stream);
      if (rc != FLCE_OK) return rc;
      if (gh) {
        FLCE_LAUNCH(K_CONVERT, launch_f32_to_bf16(gh32, static_cast<uint16_t*>(c.grad_h) + r0 * H,
                                                  static_cast<int64_t>(rows) * H, stream));
      }
      continue;
    }

    // ---- dlogits
    DlogitParams dp{};
    dp.rows = rows;
    dp.vocab = V;
    dp.s = zbuf;
    dp.lds = L.ldz;
    dp.s16 = z16;
    dp.gmax = gmax;
    dp.ldg = L.ldg;
    dp.lse = lse;
    dp.labels = lab_c;
    dp.ignore_index = p.ignore_index;
    dp.softcap = p.softcap;
    dp.inv_softcap = inv_cap;
    dp.grad_scale = p.grad_scale;
    dp.reduction = p.reduction;
    dp.hdr = hdr;
    dp.dz = dz;
    dp.ldd = L.ldd;
    dp.dzt = dzt;
    dp.ldt = L.ldt;
    FLCE_LAUNCH(K_DLOGITS, launch_dlogits(dp, stream));

    // ---- grad_h = m dz W
    if (gh) {
      GemmParams b{};
      std::memset(&b, 0, sizeof(b));
      b.M = rows;
      b.N = H;
      b.K = V;
      b.m_tiles = (rows + kBM - 1) / kBM;
      b.n_tiles = (H + kBN - 1) / kBN;
      b.k_iters = (V + kBK - 1) / kBK;
      b.group_m = std::min(b.m_tiles, 16);
      b.alpha = p.out_mult;
      b.M_valid = rows;
      b.N_valid = H;
      b.out = static_cast<uint16_t*>(c.grad_h) + r0 * H;
      b.ldo = H;
      b.status = &hdr->status;
      b.timeout_ns = timeout;
      if (simt) {
        FLCE_LAUNCH(K_GRADH_GEMM, launch_gemm_simt(EPI_BF16, dz, L.ldd, wt, L.ldwt, b, stream));
      } else {
        CUtensorMap map_dz, map_wb;
        if (!encode_bf16(&map_dz, dz, V, rows, L.ldd, kBM)) return FLCE_ERR_UNSUPPORTED;
        if (kmajor) {
          map_wb = map_wt;  // W^T [H][V]: K-major B
        } else if (!encode_bf16(&map_wb, c.W, H, V, n.ld_w, 64)) {  // W [V][H]: MN-major B
          return FLCE_ERR_UNSUPPORTED;
        }
        FLCE_LAUNCH(K_GRADH_GEMM, launch_gemm_tc(EPI_BF16, false, !kmajor, wide_for(b), &map_dz, &map_wb, nullptr, b,
                                                 std::min(b.m_tiles * b.n_tiles, sms), stream, pair && !kmajor));
      }
    }

    // ---- grad_W += m dz^T h_c
    if (gw && !simt && !kmajor) {  // dz and h_c read in place
      const AccCtx x{p.out_mult, hdr, timeout, p.flags, sms, pair, stream};
      rc = grad_W_acc_gemm(x, dz, L.ldd, rows, V, h_c, ld_hc, H, c.grad_W);
      if (rc != FLCE_OK) return rc;
    } else if (gw) {  // the debug paths: transposed copies
      if (kmajor) {
        FLCE_LAUNCH(K_TRANSPOSE_H, launch_transpose_bf16(static_cast<const uint16_t*>(c.h) + r0 * n.ld_h,
                                                         n.ld_h, rows, H, ht, L.ldht, stream));
      }
      GemmParams b{};
      std::memset(&b, 0, sizeof(b));
      b.M = V;
      b.N = H;
      b.K = rows;
      b.m_tiles = (V + kBM - 1) / kBM;
      b.n_tiles = (H + kBN - 1) / kBN;
      b.k_iters = (rows + kBK - 1) / kBK;
      b.group_m = std::min(b.m_tiles, 16);
      b.alpha = p.out_mult;
      b.M_valid = V;
      b.N_valid = H;
      b.out = c.grad_W;
      b.ldo = H;
      b.status = &hdr->status;
      b.timeout_ns = timeout;
      if (simt) {
        FLCE_LAUNCH(K_GRADW_GEMM, launch_gemm_simt(EPI_ACC_F32, dzt, L.ldt, ht, L.ldht, b, stream));
      } else {
        // dz^T [V][C] and h_c^T [H][C]: K-major A and B
        CUtensorMap map_a, map_b, map_o;
        if (!encode_bf16(&map_a, dzt, rows, V, L.ldt, kBM)) return FLCE_ERR_UNSUPPORTED;
        if (!encode_bf16(&map_b, ht, rows, H, L.ldht, kBN)) return FLCE_ERR_UNSUPPORTED;
        if (!encode_f32_out(&map_o, c.grad_W, H, V, H)) return FLCE_ERR_UNSUPPORTED;
        FLCE_LAUNCH(K_GRADW_GEMM, launch_gemm_tc(EPI_ACC_F32, false, false, wide_for(b), &map_a, &map_b, &map_o, b,
                                                 std::min(b.m_tiles * b.n_tiles, sms), stream, false));
      }
    }
  }

  if (shard) return FLCE_OK;  // the loss needs every shard's partials (flce_vp_backward)
  FLCE_LAUNCH(K_FINISH, launch_finish(hdr, p.reduction, out_loss, out_acc, stream));
  if (c.host_in) {
    if (cudaMemcpyAsync(c.loss, out_loss, sizeof(float), cudaMemcpyDeviceToHost, stream) != cudaSuccess)
      return FLCE_ERR_CUDA;
    if (c.acc && cudaMemcpyAsync(c.acc, out_acc, sizeof(float), cudaMemcpyDeviceToHost, stream) != cudaSuccess)
      return FLCE_ERR_CUDA;
  }
  return FLCE_OK;
}

// ------------------------------------------------------------ vocab-parallel
// Checks of a shard's place among the shards: offsets[0] = 0, increasing,
// offsets[S] = vocab_total, and the shard [vocab_offset, vocab_offset + V_k)
// one of the ranges.
int check_shards(int64_t vocab_offset, int64_t vocab_shard, int64_t vocab_total, int n_shards,
                 const int64_t* offsets) {
  if (vocab_total <= 0 || vocab_total >= (int64_t(1) << 31) - 512) return FLCE_ERR_ARG;
  if (vocab_offset < 0 || vocab_offset + vocab_shard > vocab_total) return FLCE_ERR_ARG;
  if (n_shards < 0) return FLCE_ERR_ARG;
  if (n_shards == 0) return FLCE_OK;  // forward: no table given
  if (n_shards > kMaxShards || offsets == nullptr) return FLCE_ERR_ARG;
  if (offsets[0] != 0 || offsets[n_shards] != vocab_total) return FLCE_ERR_ARG;
  bool mine = false;
  for (int k = 0; k < n_shards; ++k) {
    if (offsets[k + 1] <= offsets[k]) return FLCE_ERR_ARG;
    if (offsets[k] == vocab_offset && offsets[k + 1] - offsets[k] == vocab_shard) mine = true;
  }
  return mine ? FLCE_OK : FLCE_ERR_ARG;
}

struct VpLayout {
  int64_t C, slab, blocks;
  size_t off_hdr, off_bl, off_bc, off_lse, off_dz, total;
};

void make_vp_layout(const Norm& n, bool grads, VpLayout* L) {
  const flce_params& p = n.p;
  int64_t c = p.chunk_rows > 0 ? p.chunk_rows : kDefaultChunkRows;
  c = std::min<int64_t>(c, std::max<int64_t>(p.n_rows, 1));
  c = std::min<int64_t>(c, 32768);
  L->C = round_up(c, kBM);
  const int64_t want = p.vocab_slab > 0 ? p.vocab_slab : 16384;
  L->slab = round_up(std::min<int64_t>(want, round_up(p.vocab, kVTile)), kVTile);
  L->blocks = (std::max<int64_t>(p.n_rows, 1) + 31) / 32;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += (bytes + 255) / 256 * 256;
    return o;
  };
  L->off_hdr = take(sizeof(Header));
  L->off_bl = take(sizeof(double) * L->blocks);
  L->off_bc = take(sizeof(int64_t) * L->blocks);
  L->off_lse = take(sizeof(float) * std::max<int64_t>(p.n_rows, 1));
  L->off_dz = grads ? take(sizeof(uint16_t) * L->C * L->slab) : 0;
  L->total = off;
}

// Backward of one vocab shard: merge of every shard's partials into lse, loss,
// accuracy and predictions (the same on every shard), then the recompute
// backward over the shard's vocab slabs, chunk by chunk.
int run_vp_backward(const flce_params* params, int64_t vocab_offset, int64_t vocab_total, int n_shards,
                    const int64_t* offsets, const float* all_partials, const void* h, const void* W,
                    const int64_t* labels, float* loss, float* acc, int64_t* predicted, float* row_lse,
                    float* gh_acc, float* grad_W, void* wsv, size_t ws_bytes, cudaStream_t stream) {
  Norm n;
  int rc = normalise(params, &n);
  if (rc != FLCE_OK) return rc;
  const flce_params& p = n.p;
  if (p.dtype != FLCE_DTYPE_BF16) return FLCE_ERR_UNSUPPORTED;
  if (p.flags & (FLCE_FLAG_SIMT_GEMM | FLCE_FLAG_KMAJOR_BWD)) return FLCE_ERR_UNSUPPORTED;
  if (n_shards < 1) return FLCE_ERR_ARG;
  rc = check_shards(vocab_offset, p.vocab, vocab_total, n_shards, offsets);
  if (rc != FLCE_OK) return rc;
  if (!loss || !wsv || !W) return FLCE_ERR_ARG;
  if (p.n_rows > 0 && (!h || !labels || !all_partials)) return FLCE_ERR_ARG;
  if (!aligned16(wsv) || (h && !aligned16(h)) || !aligned16(W)) return FLCE_ERR_ALIGN;
  if ((gh_acc && !aligned16(gh_acc)) || (grad_W && !aligned16(grad_W))) return FLCE_ERR_ALIGN;
  const bool grads = gh_acc != nullptr || grad_W != nullptr;
  // FLCE_FLAG_VP_STORED: the forward's stored logits come first in the
  // workspace (the layout both calls compute), this call's own part after them
  const bool stored = (p.flags & FLCE_FLAG_VP_STORED) != 0;
  if (stored && (rc = check_vp_stored(p)) != FLCE_OK) return rc;
  Layout Ls{};
  if (stored) make_vp_stored_layout(n, &Ls);
  const size_t base = stored ? Ls.total : 0;
  VpLayout L;
  make_vp_layout(n, grads && !stored, &L);
  if (ws_bytes < base + L.total) return FLCE_ERR_WORKSPACE;
  int sms = 0, cc = 0;
  rc = device_info(&sms, &cc);
  if (rc != FLCE_OK) return rc;
  if (cc != 103) return FLCE_ERR_UNSUPPORTED;
  if (!load_encoder()) return FLCE_ERR_UNSUPPORTED;

  uint8_t* ws_all = static_cast<uint8_t*>(wsv);
  uint8_t* ws = ws_all + base;
  // the status word stays at the start of the workspace (flce_get_status):
  // with stored logits this call takes over the forward's header there
  Header* hdr = reinterpret_cast<Header*>(stored ? ws_all + Ls.off_hdr : ws + L.off_hdr);
  float* lse_all = reinterpret_cast<float*>(ws + L.off_lse);
  const int N = static_cast<int>(p.n_rows), H = static_cast<int>(p.hidden), V = static_cast<int>(p.vocab);
  FLCE_LAUNCH(K_PROLOGUE, launch_prologue(labels, p.n_rows, vocab_total, p.ignore_index, hdr, stream));
  VpMergeParams mp{};
  mp.rows = N;
  mp.n_shards = n_shards;
  for (int k = 0; k <= n_shards; ++k) mp.offsets[k] = static_cast<int32_t>(offsets[k]);
  mp.partials = all_partials;
  mp.ld = p.n_rows;
  mp.labels = labels;
  mp.ignore_index = p.ignore_index;
  mp.lse = lse_all;
  mp.predicted = predicted;
  mp.row_lse = row_lse;
  mp.block_loss = reinterpret_cast<double*>(ws + L.off_bl);
  mp.block_correct = reinterpret_cast<int64_t*>(ws + L.off_bc);
  mp.hdr = hdr;
  FLCE_LAUNCH(K_VP_MERGE, launch_vp_merge(mp, stream));
  FLCE_LAUNCH(K_FINISH, launch_finish(hdr, p.reduction, loss, acc, stream));
  if (!grads || N == 0) return FLCE_OK;

  CUtensorMap map_h, map_w, map_w_pair;
  const bool pair = (p.flags & FLCE_FLAG_CTA_PAIR) != 0;
  if (!encode_bf16(&map_h, h, H, N, n.ld_h, kBM)) return FLCE_ERR_UNSUPPORTED;
  if (!encode_bf16(&map_w, W, H, V, n.ld_w, kBN)) return FLCE_ERR_UNSUPPORTED;
  if (pair && !encode_bf16(&map_w_pair, W, H, V, n.ld_w, kBN / 2)) return FLCE_ERR_UNSUPPORTED;
  const uint64_t timeout = p.timeout_ns > 0 ? static_cast<uint64_t>(p.timeout_ns) : kDefaultTimeoutNs;
  if (stored) {
    // per chunk of C rows: dlogits from the kept logits (labels relative to
    // the shard), then grad_h_partial += m dz W_k and grad_W_k += m dz^T h_c,
    // as the fused path does
    uint16_t* z16 = reinterpret_cast<uint16_t*>(ws_all + Ls.off_z);
    float* gmax = reinterpret_cast<float*>(ws_all + Ls.off_gmax);
    uint16_t* dz = reinterpret_cast<uint16_t*>(ws_all + Ls.off_dz);
    const AccCtx x{p.out_mult, hdr, timeout, p.flags, sms, pair, stream};
    for (int64_t r0 = 0; r0 < p.n_rows; r0 += Ls.C) {
      const int rows = static_cast<int>(std::min<int64_t>(Ls.C, p.n_rows - r0));
      DlogitParams dp{};
      dp.rows = rows;
      dp.vocab = V;
      dp.s16 = z16 + r0 * Ls.ldz;
      dp.lds = Ls.ldz;
      dp.gmax = gmax + r0 * Ls.ldg;
      dp.ldg = Ls.ldg;
      dp.lse = lse_all + r0;
      dp.labels = labels + r0;
      dp.label_offset = vocab_offset;
      dp.ignore_index = p.ignore_index;
      dp.softcap = p.softcap;
      dp.inv_softcap = p.softcap > 0.f ? 1.f / p.softcap : 0.f;
      dp.grad_scale = p.grad_scale;
      dp.reduction = p.reduction;
      dp.hdr = hdr;
      dp.dz = dz;
      dp.ldd = Ls.ldd;
      FLCE_LAUNCH(K_DLOGITS, launch_dlogits(dp, stream));
      if (gh_acc) {
        rc = grad_h_acc_gemm(x, dz, Ls.ldd, rows, V, static_cast<const uint16_t*>(W), n.ld_w, H, gh_acc + r0 * H, 16);
        if (rc != FLCE_OK) return rc;
      }
      if (grad_W) {
        rc = grad_W_acc_gemm(x, dz, Ls.ldd, rows, V, static_cast<const uint16_t*>(h) + r0 * n.ld_h, n.ld_h, H, grad_W);
        if (rc != FLCE_OK) return rc;
      }
    }
    return FLCE_OK;
  }
  for (int64_t r0 = 0; r0 < p.n_rows; r0 += L.C) {
    SlabArgs sa;
    sa.rows = static_cast<int>(std::min<int64_t>(L.C, p.n_rows - r0));
    sa.H = H;
    sa.V = V;
    sa.slab = static_cast<int>(L.slab);
    sa.col_base = static_cast<int>(vocab_offset);
    sa.h_row0 = static_cast<int>(r0);
    sa.map_hc = &map_h;
    sa.map_w = &map_w;
    sa.map_w_pair = pair ? &map_w_pair : nullptr;
    sa.h_c = static_cast<const uint16_t*>(h) + r0 * n.ld_h;
    sa.ld_hc = n.ld_h;
    sa.W = static_cast<const uint16_t*>(W);
    sa.ld_w = n.ld_w;
    sa.labels = labels + r0;
    sa.lse = lse_all + r0;
    sa.hdr = hdr;
    sa.dz = reinterpret_cast<uint16_t*>(ws + L.off_dz);
    sa.gh_acc = gh_acc ? gh_acc + r0 * H : nullptr;
    sa.grad_W = grad_W;
    sa.p = &p;
    sa.inv_cap = p.softcap > 0.f ? 1.f / p.softcap : 0.f;
    sa.timeout = timeout;
    sa.sms = sms;
    rc = recompute_slabs(sa, stream);
    if (rc != FLCE_OK) return rc;
  }
  return FLCE_OK;
}

// fp32 operands (the pages' fp32 parity and convergence runs): tcgen05
// kind::tf32 GEMMs on K-major operands, fp32 dlogits with an fp32 transposed
// copy, fp32 transposes of W and h_c, grad_h written in fp32 by bulk stores.
int run_f32(const Norm& n, const Call& c) {
  const flce_params& p = n.p;
  const bool gh = c.mode == FLCE_MODE_FORWARD_BACKWARD && c.grad_h != nullptr;
  const bool gw = c.mode == FLCE_MODE_FORWARD_BACKWARD && c.grad_W != nullptr;
  if (!c.loss || !c.ws || !c.W) return FLCE_ERR_ARG;
  if (p.n_rows > 0 && (!c.h || !c.labels)) return FLCE_ERR_ARG;
  if (!aligned16(c.ws) || (!c.host_in && c.h && !aligned16(c.h)) || !aligned16(c.W)) return FLCE_ERR_ALIGN;
  if ((gh && !aligned16(c.grad_h)) || (gw && !aligned16(c.grad_W))) return FLCE_ERR_ALIGN;
  if (p.flags & (FLCE_FLAG_SIMT_GEMM | FLCE_FLAG_RECOMPUTE)) return FLCE_ERR_UNSUPPORTED;
  Layout L;
  make_layout(n, !c.host_in ? c.mode
                             : c.mode == FLCE_MODE_CE_ONLY ? FLCE_MODE_CE_ONLY_HOST : FLCE_MODE_FORWARD_BACKWARD_HOST,
              gh, gw, &L);
  if (c.ws_bytes < L.total) return FLCE_ERR_WORKSPACE;
  int sms = 0, cc = 0;
  int rc = device_info(&sms, &cc);
  if (rc != FLCE_OK) return rc;
  if (cc != 103) return FLCE_ERR_UNSUPPORTED;
  if (!load_encoder()) return FLCE_ERR_UNSUPPORTED;

  cudaStream_t stream = c.stream;
  uint8_t* ws = static_cast<uint8_t*>(c.ws);
  Header* hdr = reinterpret_cast<Header*>(ws + L.off_hdr);
  float* pmax = reinterpret_cast<float*>(ws + L.off_pmax);
  float* psum = reinterpret_cast<float*>(ws + L.off_psum);
  int32_t* pidx = reinterpret_cast<int32_t*>(ws + L.off_pidx);
  float* tgt = reinterpret_cast<float*>(ws + L.off_tgt);
  float* lse = reinterpret_cast<float*>(ws + L.off_lse);
  float* zbuf = L.need_z ? reinterpret_cast<float*>(ws + L.off_z) : nullptr;
  float* dz = L.need_dz ? reinterpret_cast<float*>(ws + L.off_dz) : nullptr;
  float* dzt = L.need_dzt ? reinterpret_cast<float*>(ws + L.off_dzt) : nullptr;
  float* wt = L.need_wt ? reinterpret_cast<float*>(ws + L.off_wt) : nullptr;
  float* ht = L.need_ht ? reinterpret_cast<float*>(ws + L.off_ht) : nullptr;
  const uint64_t timeout = p.timeout_ns > 0 ? static_cast<uint64_t>(p.timeout_ns) : kDefaultTimeoutNs;
  const int N = static_cast<int>(p.n_rows), H = static_cast<int>(p.hidden), V = static_cast<int>(p.vocab);
  const float inv_cap = p.softcap > 0.f ? 1.f / p.softcap : 0.f;
  const float* h = static_cast<const float*>(c.h);
  const float* W = static_cast<const float*>(c.W);
  constexpr int kSlice = kBK / 2;  // fp32 elements per 128-byte K slice

  // host inputs: staged as in run(), with 4-byte elements
  const int64_t* labels = c.labels;
  float* out_loss = c.loss;
  float* out_acc = c.acc;
  HostStaging hs;
  if (c.host_in) {
    labels = reinterpret_cast<const int64_t*>(ws + L.off_labels);
    out_loss = reinterpret_cast<float*>(ws + L.off_out);
    out_acc = out_loss + 1;
    if (p.n_rows > 0 &&
        cudaMemcpyAsync(const_cast<int64_t*>(labels), c.labels, sizeof(int64_t) * p.n_rows, cudaMemcpyHostToDevice,
                        stream) != cudaSuccess)
      return FLCE_ERR_CUDA;
    if (!hs.init(ws + L.off_hstage, L.hstage_bytes, c.h, n.ld_h, H, 4, p.n_rows, L.C, stream, c.copy_stream))
      return FLCE_ERR_CUDA;
  }

  FLCE_LAUNCH(K_PROLOGUE, launch_prologue(labels, p.n_rows, p.vocab, p.ignore_index, hdr, stream));
  // Three-pass tf32: every GEMM operand as hi = tf32(x) and lo = x - hi.
  const bool split = L.split;
  float* w_hi = split ? reinterpret_cast<float*>(ws + L.off_whi) : nullptr;
  float* w_lo = split ? reinterpret_cast<float*>(ws + L.off_wlo) : nullptr;
  float* h_hi = split ? reinterpret_cast<float*>(ws + L.off_hhi) : nullptr;
  float* h_lo = split ? reinterpret_cast<float*>(ws + L.off_hlo) : nullptr;
  float* wt_lo = split && L.need_wt ? reinterpret_cast<float*>(ws + L.off_wtlo) : nullptr;
  float* ht_lo = split && L.need_ht ? reinterpret_cast<float*>(ws + L.off_htlo) : nullptr;
  float* dz_lo = split && L.need_dz ? reinterpret_cast<float*>(ws + L.off_dzlo) : nullptr;
  float* dzt_lo = split && L.need_dzt ? reinterpret_cast<float*>(ws + L.off_dztlo) : nullptr;
  const bool wide_ok = !split;  // the split runs on 128-row tiles
  CUtensorMap map_h, map_w, map_wt, map_w_lo, map_wt_lo;
  if (N > 0) {
    if (!c.host_in && !split && !encode_f32_in(&map_h, h, H, N, n.ld_h, kBM)) return FLCE_ERR_UNSUPPORTED;
    if (split) {
      FLCE_LAUNCH(K_SPLIT, launch_split_f32(W, n.ld_w, V, H, w_hi, w_lo, H, stream));
      if (!encode_f32_in(&map_w, w_hi, H, V, H, kBN)) return FLCE_ERR_UNSUPPORTED;
      if (!encode_f32_in(&map_w_lo, w_lo, H, V, H, kBN)) return FLCE_ERR_UNSUPPORTED;
    } else if (!encode_f32_in(&map_w, W, H, V, n.ld_w, kBN)) {
      return FLCE_ERR_UNSUPPORTED;
    }
  }
  if (L.need_wt && N > 0) {
    FLCE_LAUNCH(K_TRANSPOSE_W, launch_transpose_f32(W, n.ld_w, V, H, wt, L.ldwt, stream, wt_lo));
    if (!encode_f32_in(&map_wt, wt, V, H, L.ldwt, kBN)) return FLCE_ERR_UNSUPPORTED;
    if (split && !encode_f32_in(&map_wt_lo, wt_lo, V, H, L.ldwt, kBN)) return FLCE_ERR_UNSUPPORTED;
  }
  for (int64_t r0 = 0; r0 < p.n_rows; r0 += L.C) {
    const int rows = static_cast<int>(std::min<int64_t>(L.C, p.n_rows - r0));
    const int64_t* lab_c = labels + r0;
    // this chunk's rows of h: the caller's array or the staging buffer
    const float* h_c = h + r0 * n.ld_h;
    int64_t ld_hc = n.ld_h;
    int h_row0 = static_cast<int>(r0);
    CUtensorMap map_hc = map_h, map_hc_lo;
    if (c.host_in) {
      h_c = static_cast<const float*>(hs.wait_chunk(r0 / L.C));
      if (!h_c) return FLCE_ERR_CUDA;
      ld_hc = H;
      h_row0 = 0;
      if (!split && !encode_f32_in(&map_hc, h_c, H, rows, H, kBM)) return FLCE_ERR_UNSUPPORTED;
    }
    if (split) {  // this chunk's rows as hi / lo
      FLCE_LAUNCH(K_SPLIT, launch_split_f32(h_c, ld_hc, rows, H, h_hi, h_lo, H, stream));
      if (!encode_f32_in(&map_hc, h_hi, H, rows, H, kBM)) return FLCE_ERR_UNSUPPORTED;
      if (!encode_f32_in(&map_hc_lo, h_lo, H, rows, H, kBM)) return FLCE_ERR_UNSUPPORTED;
      h_row0 = 0;
    }
    GemmParams g{};
    std::memset(&g, 0, sizeof(g));
    g.M = rows;
    g.N = V;
    g.K = H;
    g.m_tiles = (rows + kBM - 1) / kBM;
    g.n_tiles = static_cast<int>(L.n_vtiles);
    g.k_iters = (H + kSlice - 1) / kSlice;
    g.group_m = std::min(g.m_tiles, 16);
    g.a_row0 = h_row0;
    g.alpha = p.out_mult;
    g.M_valid = rows;
    g.N_valid = V;
    g.softcap = p.softcap;
    g.inv_softcap = inv_cap;
    g.labels = lab_c;
    g.ignore_index = p.ignore_index;
    g.part_max = pmax;
    g.part_sum = psum;
    g.part_idx = pidx;
    g.tgt = tgt;
    g.ldp = static_cast<int>(L.ldp);
    g.zbuf = zbuf;
    g.ldz = L.ldz;
    g.status = &hdr->status;
    g.timeout_ns = timeout;
    g.debug_flags = p.flags;
    g.no_argmax = c.predicted == nullptr ? 1 : 0;
    const bool store = L.need_z;
    g.store_hint = store ? 1 : 0;
    CUtensorMap map_z;
    if (store && !encode_f32_out(&map_z, zbuf, L.ldz, rows, L.ldz)) return FLCE_ERR_UNSUPPORTED;
    FLCE_LAUNCH(K_FWD_GEMM, launch_gemm_tc_tf32(store ? EPI_STATS_STORE : EPI_STATS,
                                                wide_ok && pick_wide(p.flags, g, sms), &map_hc, &map_w,
                                                store ? &map_z : nullptr, g, std::min(g.m_tiles * g.n_tiles, sms),
                                                stream, split ? &map_hc_lo : nullptr, split ? &map_w_lo : nullptr));
    MergeParams mp{};
    mp.rows = rows;
    mp.n_vtiles = static_cast<int>(L.n_vtiles);
    mp.ldp = static_cast<int>(L.ldp);
    mp.part_max = pmax;
    mp.part_sum = psum;
    mp.part_idx = pidx;
    mp.tgt = tgt;
    mp.labels = lab_c;
    mp.ignore_index = p.ignore_index;
    mp.lse = lse;
    mp.predicted = c.predicted ? c.predicted + r0 : nullptr;
    mp.row_lse = c.row_lse ? c.row_lse + r0 : nullptr;
    mp.block_loss = reinterpret_cast<double*>(ws + L.off_bl);
    mp.block_correct = reinterpret_cast<int64_t*>(ws + L.off_bc);
    mp.hdr = hdr;
    FLCE_LAUNCH(K_MERGE, launch_merge(mp, stream));
    if (!gh && !gw) continue;

    DlogitParams dp{};
    dp.rows = rows;
    dp.vocab = V;
    dp.s = zbuf;
    dp.lds = L.ldz;
    dp.lse = lse;
    dp.labels = lab_c;
    dp.ignore_index = p.ignore_index;
    dp.softcap = p.softcap;
    dp.inv_softcap = inv_cap;
    dp.grad_scale = p.grad_scale;
    dp.reduction = p.reduction;
    dp.hdr = hdr;
    dp.dz32 = gh ? dz : nullptr;
    dp.ldd = L.ldd;
    dp.dzt32 = gw ? dzt : nullptr;
    dp.ldt = L.ldt;
    dp.dz32_lo = gh ? dz_lo : nullptr;
    dp.dzt32_lo = gw ? dzt_lo : nullptr;
    FLCE_LAUNCH(K_DLOGITS, launch_dlogits(dp, stream));

    if (gh) {  // grad_h_c = m dz W: A = dz [C][V], B = W^T [H][V], fp32 output
      GemmParams b{};
      std::memset(&b, 0, sizeof(b));
      b.M = rows;
      b.N = H;
      b.K = V;
      b.m_tiles = (rows + kBM - 1) / kBM;
      b.n_tiles = (H + kBN - 1) / kBN;
      b.k_iters = (V + kSlice - 1) / kSlice;
      b.group_m = std::min(b.m_tiles, 16);
      b.alpha = p.out_mult;
      b.M_valid = rows;
      b.N_valid = H;
      b.status = &hdr->status;
      b.timeout_ns = timeout;
      CUtensorMap map_a, map_o, map_a_lo;
      if (!encode_f32_in(&map_a, dz, V, rows, L.ldd, kBM)) return FLCE_ERR_UNSUPPORTED;
      if (split && !encode_f32_in(&map_a_lo, dz_lo, V, rows, L.ldd, kBM)) return FLCE_ERR_UNSUPPORTED;
      if (!encode_f32_out(&map_o, static_cast<float*>(c.grad_h) + r0 * H, H, rows, H)) return FLCE_ERR_UNSUPPORTED;
      FLCE_LAUNCH(K_GRADH_GEMM, launch_gemm_tc_tf32(EPI_F32, wide_ok && pick_wide(p.flags, b, sms), &map_a, &map_wt,
                                                    &map_o, b, std::min(b.m_tiles * b.n_tiles, sms), stream,
                                                    split ? &map_a_lo : nullptr, split ? &map_wt_lo : nullptr));
    }
    if (gw) {  // grad_W += m dz^T h_c: A = dz^T [V][C], B = h_c^T [H][C]
      FLCE_LAUNCH(K_TRANSPOSE_H, launch_transpose_f32(h_c, ld_hc, rows, H, ht, L.ldht, stream, ht_lo));
      GemmParams b{};
      std::memset(&b, 0, sizeof(b));
      b.M = V;
      b.N = H;
      b.K = rows;
      b.m_tiles = (V + kBM - 1) / kBM;
      b.n_tiles = (H + kBN - 1) / kBN;
      b.k_iters = (rows + kSlice - 1) / kSlice;
      b.group_m = std::min(b.m_tiles, 16);
      b.alpha = p.out_mult;
      b.M_valid = V;
      b.N_valid = H;
      b.status = &hdr->status;
      b.timeout_ns = timeout;
      CUtensorMap map_a, map_b, map_o, map_a_lo, map_b_lo;
      if (!encode_f32_in(&map_a, dzt, rows, V, L.ldt, kBM)) return FLCE_ERR_UNSUPPORTED;
      if (!encode_f32_in(&map_b, ht, rows, H, L.ldht, kBN)) return FLCE_ERR_UNSUPPORTED;
      if (split && !encode_f32_in(&map_a_lo, dzt_lo, rows, V, L.ldt, kBM)) return FLCE_ERR_UNSUPPORTED;
      if (split && !encode_f32_in(&map_b_lo, ht_lo, rows, H, L.ldht, kBN)) return FLCE_ERR_UNSUPPORTED;
      if (!encode_f32_out(&map_o, c.grad_W, H, V, H)) return FLCE_ERR_UNSUPPORTED;
      FLCE_LAUNCH(K_GRADW_GEMM, launch_gemm_tc_tf32(EPI_ACC_F32, wide_ok && pick_wide(p.flags, b, sms), &map_a, &map_b,
                                                    &map_o, b, std::min(b.m_tiles * b.n_tiles, sms), stream,
                                                    split ? &map_a_lo : nullptr, split ? &map_b_lo : nullptr));
    }
  }
  FLCE_LAUNCH(K_FINISH, launch_finish(hdr, p.reduction, out_loss, out_acc, stream));
  if (c.host_in) {
    if (cudaMemcpyAsync(c.loss, out_loss, sizeof(float), cudaMemcpyDeviceToHost, stream) != cudaSuccess)
      return FLCE_ERR_CUDA;
    if (c.acc && cudaMemcpyAsync(c.acc, out_acc, sizeof(float), cudaMemcpyDeviceToHost, stream) != cudaSuccess)
      return FLCE_ERR_CUDA;
  }
  return FLCE_OK;
}

// Cross-entropy on materialised logits: prologue, then per chunk the tile
// statistics, the merge and (when asked) the gradient, then the scalars.
int run_ce(const flce_params* params, const void* logits, int dtype, int64_t ldx, const int64_t* labels,
           float* loss, float* acc, int64_t* predicted, float* row_loss, const float* row_scale, void* grad,
           void* wsv, size_t ws_bytes, cudaStream_t stream) {
  Norm n;
  int rc = normalise(params, &n, false);
  if (rc != FLCE_OK) return rc;
  const flce_params& p = n.p;
  if (dtype != FLCE_DTYPE_BF16 && dtype != FLCE_DTYPE_F32) return FLCE_ERR_ARG;
  if (!loss || !wsv) return FLCE_ERR_ARG;
  if (p.n_rows > 0 && (!logits || !labels)) return FLCE_ERR_ARG;
  if (ldx < p.vocab) return FLCE_ERR_ARG;
  if (!aligned16(wsv)) return FLCE_ERR_ALIGN;
  Layout L;
  make_layout(n, FLCE_MODE_CROSS_ENTROPY, false, false, &L);
  if (ws_bytes < L.total) return FLCE_ERR_WORKSPACE;
  int sms = 0, cc = 0;
  rc = device_info(&sms, &cc);
  if (rc != FLCE_OK) return rc;
  if (cc != 103) return FLCE_ERR_UNSUPPORTED;

  uint8_t* ws = static_cast<uint8_t*>(wsv);
  Header* hdr = reinterpret_cast<Header*>(ws + L.off_hdr);
  const size_t esz = dtype == FLCE_DTYPE_BF16 ? 2 : 4;
  const bool vec_ok = aligned16(logits) && (grad == nullptr || aligned16(grad)) && (ldx * esz) % 16 == 0;

  FLCE_LAUNCH(K_PROLOGUE, launch_prologue(labels, p.n_rows, p.vocab, p.ignore_index, hdr, stream));
  for (int64_t r0 = 0; r0 < p.n_rows; r0 += L.C) {
    const int rows = static_cast<int>(std::min<int64_t>(L.C, p.n_rows - r0));
    CeParams cp{};
    cp.rows = rows;
    cp.vocab = static_cast<int>(p.vocab);
    cp.n_vtiles = static_cast<int>(L.n_vtiles);
    cp.ldp = static_cast<int>(L.ldp);
    cp.dtype = dtype;
    cp.vec_ok = vec_ok ? 1 : 0;
    cp.logits = static_cast<const uint8_t*>(logits) + r0 * ldx * esz;
    cp.ldx = ldx;
    cp.grad = grad ? static_cast<uint8_t*>(grad) + r0 * ldx * esz : nullptr;
    cp.ldg = ldx;
    cp.labels = labels + r0;
    cp.ignore_index = p.ignore_index;
    cp.out_mult = p.out_mult;
    cp.softcap = p.softcap;
    cp.inv_softcap = p.softcap > 0.f ? 1.f / p.softcap : 0.f;
    cp.grad_scale = p.grad_scale;
    cp.reduction = p.reduction;
    cp.row_scale = row_scale ? row_scale + r0 : nullptr;
    cp.part_max = reinterpret_cast<float*>(ws + L.off_pmax);
    cp.part_sum = reinterpret_cast<float*>(ws + L.off_psum);
    cp.part_idx = reinterpret_cast<int32_t*>(ws + L.off_pidx);
    cp.tgt = reinterpret_cast<float*>(ws + L.off_tgt);
    cp.lse = reinterpret_cast<float*>(ws + L.off_lse);
    cp.hdr = hdr;
    FLCE_LAUNCH(K_CE_STATS, launch_ce_stats(cp, stream));

    MergeParams mp{};
    mp.rows = rows;
    mp.n_vtiles = static_cast<int>(L.n_vtiles);
    mp.ldp = static_cast<int>(L.ldp);
    mp.part_max = cp.part_max;
    mp.part_sum = cp.part_sum;
    mp.part_idx = cp.part_idx;
    mp.tgt = cp.tgt;
    mp.labels = labels + r0;
    mp.ignore_index = p.ignore_index;
    mp.lse = reinterpret_cast<float*>(ws + L.off_lse);
    mp.predicted = predicted ? predicted + r0 : nullptr;
    mp.row_lse = nullptr;
    mp.row_loss = row_loss ? row_loss + r0 : nullptr;
    mp.block_loss = reinterpret_cast<double*>(ws + L.off_bl);
    mp.block_correct = reinterpret_cast<int64_t*>(ws + L.off_bc);
    mp.hdr = hdr;
    FLCE_LAUNCH(K_MERGE, launch_merge(mp, stream));

    if (grad) FLCE_LAUNCH(K_CE_GRAD, launch_ce_grad(cp, stream));
  }
  FLCE_LAUNCH(K_FINISH, launch_finish(hdr, p.reduction, loss, acc, stream));
  return FLCE_OK;
}

}  // namespace

extern "C" {

void flce_default_params(flce_params* p) {
  if (!p) return;
  std::memset(p, 0, sizeof(*p));
  p->softcap = 0.f;
  p->out_mult = 1.f;
  p->ignore_index = -100;
  p->reduction = FLCE_REDUCTION_MEAN;
  p->grad_scale = 1.f;
}

size_t flce_workspace_size(const flce_params* p, int mode, int need_grad_h, int need_grad_W) {
  Norm n;
  if (mode < FLCE_MODE_CE_ONLY || mode > FLCE_MODE_CE_ONLY_HOST) return 0;
  if (normalise(p, &n, mode != FLCE_MODE_CROSS_ENTROPY) != FLCE_OK) return 0;
  Layout L;
  make_layout(n, mode, need_grad_h != 0, need_grad_W != 0, &L);
  return L.total;
}

int64_t flce_chunk_rows(const flce_params* p, int mode, int need_grad_h, int need_grad_W) {
  Norm n;
  if (mode < FLCE_MODE_CE_ONLY || mode > FLCE_MODE_CE_ONLY_HOST) return 0;
  if (normalise(p, &n, mode != FLCE_MODE_CROSS_ENTROPY) != FLCE_OK) return 0;
  Layout L;
  make_layout(n, mode, need_grad_h != 0, need_grad_W != 0, &L);
  return L.C;
}

int flce_ce_only(const flce_params* p, const void* h, const void* W, const int64_t* labels, float* loss,
                 float* token_accuracy, void* workspace, size_t workspace_bytes, void* stream) {
  Call c{FLCE_MODE_CE_ONLY, h, W, labels, loss, token_accuracy, nullptr, nullptr, nullptr, nullptr,
         workspace, workspace_bytes, static_cast<cudaStream_t>(stream)};
  return run(p, c);
}

int flce_forward(const flce_params* p, const void* h, const void* W, const int64_t* labels, float* loss,
                 float* token_accuracy, int64_t* predicted, float* row_lse, void* workspace, size_t workspace_bytes,
                 void* stream) {
  Call c{FLCE_MODE_FORWARD, h, W, labels, loss, token_accuracy, predicted, row_lse, nullptr, nullptr,
         workspace, workspace_bytes, static_cast<cudaStream_t>(stream)};
  return run(p, c);
}

int flce_forward_backward(const flce_params* p, const void* h, const void* W, const int64_t* labels, float* loss,
                          float* token_accuracy, int64_t* predicted, void* grad_h, float* grad_W, void* workspace,
                          size_t workspace_bytes, void* stream) {
  Call c{FLCE_MODE_FORWARD_BACKWARD, h, W, labels, loss, token_accuracy, predicted, nullptr, grad_h, grad_W,
         workspace, workspace_bytes, static_cast<cudaStream_t>(stream)};
  return run(p, c);
}

int flce_forward_backward_from_host(const flce_params* p, const void* h_host, const void* W,
                                   const int64_t* labels_host, float* loss_host, float* token_accuracy_host,
                                   int64_t* predicted, void* grad_h, float* grad_W, void* workspace,
                                   size_t workspace_bytes, void* stream, void* copy_stream) {
  Call c{FLCE_MODE_FORWARD_BACKWARD, h_host, W, labels_host, loss_host, token_accuracy_host, predicted, nullptr,
         grad_h, grad_W, workspace, workspace_bytes, static_cast<cudaStream_t>(stream)};
  c.host_in = true;
  c.copy_stream = static_cast<cudaStream_t>(copy_stream);
  return run(p, c);
}

int flce_ce_only_from_host(const flce_params* p, const void* h_host, const void* W, const int64_t* labels_host,
                           float* loss_host, float* token_accuracy_host, void* workspace, size_t workspace_bytes,
                           void* stream, void* copy_stream) {
  Call c{FLCE_MODE_CE_ONLY, h_host, W, labels_host, loss_host, token_accuracy_host, nullptr, nullptr, nullptr,
         nullptr, workspace, workspace_bytes, static_cast<cudaStream_t>(stream)};
  c.host_in = true;
  c.copy_stream = static_cast<cudaStream_t>(copy_stream);
  return run(p, c);
}

size_t flce_vp_workspace_size(const flce_params* p, int backward, int need_grad_h, int need_grad_W) {
  Norm n;
  if (normalise(p, &n) != FLCE_OK) return 0;
  if (n.p.flags & FLCE_FLAG_VP_STORED) {  // one size for both calls: the stored logits, then the backward's part
    if (check_vp_stored(n.p) != FLCE_OK) return 0;
    Layout Ls;
    make_vp_stored_layout(n, &Ls);
    VpLayout L;
    make_vp_layout(n, false, &L);
    return Ls.total + L.total;
  }
  if (!backward) {
    Layout L;
    make_layout(n, FLCE_MODE_CE_ONLY, false, false, &L);
    return L.total;
  }
  VpLayout L;
  make_vp_layout(n, need_grad_h != 0 || need_grad_W != 0, &L);
  return L.total;
}

int flce_vp_forward(const flce_params* p, int64_t vocab_offset, int64_t vocab_total, const void* h,
                    const void* W_shard, const int64_t* labels, float* partials, void* workspace,
                    size_t workspace_bytes, void* stream) {
  if (!p || (!partials && p->n_rows > 0)) return FLCE_ERR_ARG;
  const int rc = check_shards(vocab_offset, p->vocab, vocab_total, 0, nullptr);
  if (rc != FLCE_OK) return rc;
  if (p->dtype != FLCE_DTYPE_BF16 || (p->flags & FLCE_FLAG_SIMT_GEMM)) return FLCE_ERR_UNSUPPORTED;
  const bool stored = (p->flags & FLCE_FLAG_VP_STORED) != 0;
  if (stored && check_vp_stored(*p) != FLCE_OK) return FLCE_ERR_ARG;
  Call c{FLCE_MODE_CE_ONLY, h, W_shard, labels, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
         workspace, workspace_bytes, static_cast<cudaStream_t>(stream)};
  c.vocab_offset = vocab_offset;
  c.vocab_total = vocab_total;
  c.shard_partials = partials;  // NULL only with no rows, which write none
  c.shard_call = true;
  c.vp_stored = stored;
  return run(p, c);
}

int flce_vp_backward(const flce_params* p, int64_t vocab_offset, int64_t vocab_total, int n_shards,
                     const int64_t* shard_offsets, const float* all_partials, const void* h, const void* W_shard,
                     const int64_t* labels, float* loss, float* token_accuracy, int64_t* predicted,
                     float* row_lse, float* grad_h_partial, float* grad_W_shard, void* workspace,
                     size_t workspace_bytes, void* stream) {
  return run_vp_backward(p, vocab_offset, vocab_total, n_shards, shard_offsets, all_partials, h, W_shard, labels,
                         loss, token_accuracy, predicted, row_lse, grad_h_partial, grad_W_shard, workspace,
                         workspace_bytes, static_cast<cudaStream_t>(stream));
}

int flce_cross_entropy(const flce_params* p, const void* logits, int logits_dtype, int64_t ld_logits,
                       const int64_t* labels, float* loss, float* token_accuracy, int64_t* predicted,
                       float* row_loss, const float* row_scale, void* grad_logits, void* workspace,
                       size_t workspace_bytes, void* stream) {
  return run_ce(p, logits, logits_dtype, ld_logits, labels, loss, token_accuracy, predicted, row_loss, row_scale,
                grad_logits, workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
}

int flce_scale_gradient(const void* x, int x_dtype, void* y, int y_dtype, int64_t n, const float* scale,
                        void* stream_handle) {
  const bool dt_ok = (x_dtype == FLCE_DTYPE_BF16 || x_dtype == FLCE_DTYPE_F32) &&
                     (y_dtype == FLCE_DTYPE_BF16 || y_dtype == FLCE_DTYPE_F32);
  if (n < 0 || !dt_ok) return FLCE_ERR_ARG;
  if (n == 0) return FLCE_OK;
  if (!x || !y) return FLCE_ERR_ARG;
  const uintptr_t x0 = reinterpret_cast<uintptr_t>(x), y0 = reinterpret_cast<uintptr_t>(y);
  const uintptr_t xb = static_cast<uintptr_t>(n) * (x_dtype == FLCE_DTYPE_F32 ? 4u : 2u);
  const uintptr_t yb = static_cast<uintptr_t>(n) * (y_dtype == FLCE_DTYPE_F32 ? 4u : 2u);
  const bool overlap = x0 < y0 + yb && y0 < x0 + xb;
  if (overlap && !(x0 == y0 && x_dtype == y_dtype)) return FLCE_ERR_ARG;
  int sms = 0, cc = 0;
  const int rc = device_info(&sms, &cc);
  if (rc != FLCE_OK) return rc;
  if (cc != 103) return FLCE_ERR_UNSUPPORTED;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_handle);
  FLCE_LAUNCH(K_SCALE, launch_scale_convert(x, x_dtype == FLCE_DTYPE_F32, y, y_dtype == FLCE_DTYPE_F32, n, scale,
                                            sms, stream));
  return FLCE_OK;
}

int flce_get_status(const void* workspace, void* stream, int32_t* status) {
  if (!workspace || !status) return FLCE_ERR_ARG;
  int32_t v = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess) return FLCE_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return FLCE_ERR_CUDA;
  *status = v;
  return FLCE_OK;
}

const char* flce_status_string(int code) {
  switch (code) {
    case FLCE_OK: return "ok";
    case FLCE_ERR_ARG: return "invalid argument";
    case FLCE_ERR_ALIGN: return "misaligned pointer, stride or hidden size";
    case FLCE_ERR_WORKSPACE: return "workspace too small";
    case FLCE_ERR_UNSUPPORTED: return "unsupported device or tensor layout";
    case FLCE_ERR_CUDA: return "CUDA runtime error";
    case FLCE_ERR_LABEL: return "label outside [0, V) that is not ignore_index";
    case FLCE_ERR_TIMEOUT: return "bounded device wait timed out";
    case FLCE_ERR_LABEL | FLCE_ERR_TIMEOUT: return "bad label and device wait timed out";
    case FLCE_ERR_NONFINITE: return "non-finite log-sum-exp in some row (inf or NaN inputs)";
    default: return "unknown status";
  }
}

int64_t flce_launch_count(void) { return g_launches.load(); }

int flce_profile_begin(int enable) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  for (auto& r : g_prof) {
    cudaEventDestroy(r.start);
    cudaEventDestroy(r.stop);
  }
  g_prof.clear();
  g_prof_on = enable != 0;
  return FLCE_OK;
}

int flce_profile_read(int64_t* launches, double* total_ms, int n) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  for (int i = 0; i < n; ++i) {
    if (launches) launches[i] = 0;
    if (total_ms) total_ms[i] = 0.0;
  }
  int rc = FLCE_NUM_KERNELS;
  for (auto& r : g_prof) {
    float ms = 0.f;
    if (cudaEventSynchronize(r.stop) != cudaSuccess || cudaEventElapsedTime(&ms, r.start, r.stop) != cudaSuccess) {
      rc = -FLCE_ERR_CUDA;
    }
    if (r.kernel >= 0 && r.kernel < n) {
      if (launches) launches[r.kernel] += 1;
      if (total_ms) total_ms[r.kernel] += ms;
    }
    cudaEventDestroy(r.start);
    cudaEventDestroy(r.stop);
  }
  g_prof.clear();
  return rc;
}

const char* flce_kernel_name(int id) {
  if (id < 0 || id >= FLCE_NUM_KERNELS) return "unknown";
  return kKernelNames[id];
}

}  // extern "C"
