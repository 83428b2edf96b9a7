// Internal interface between the host engine and the kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "flce.h"

namespace flce {

// Tile of one tensor-core MMA: 128 rows of D (one TMEM lane per row), 256
// columns (fp32 accumulator = 256 TMEM columns), 64-element K slices (one
// 128-byte swizzle row per operand row). A CTA owns one such tile with two
// accumulator buffers (all 512 columns, kStages-deep ring), or two stacked
// (256 x 256, one buffer, a 3-stage ring of the same bytes).
constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBK = 64;
constexpr int kStages = 4;
constexpr int kGemmThreads = 192;  // warp 0: TMA, warp 1: MMA + TMEM owner, warps 2-5: epilogue
// Threads of the tensor-core GEMM: 128-row tiles (tmh = 1) have four epilogue
// warps, 256-row tiles (tmh = 2) eight.
constexpr int gemm_threads(int tmh) { return tmh == 2 ? 320 : kGemmThreads; }
constexpr int kAStageBytes = kBM * kBK * 2;
constexpr int kBStageBytes = kBN * kBK * 2;
// Per epilogue warp: two 4 KB staging buffers for a 32 x 32 fp32 sub-tile that a
// TMA bulk store (stored logits) or bulk reduce-add (fp32 gradients) sends out.
constexpr int kStageBufBytes = 32 * 32 * 4;
constexpr int kEpiStagingBytes = 4 * 2 * kStageBufBytes;
constexpr int kGemmSmemBytes =
    kStages * (kAStageBytes + kBStageBytes) + kEpiStagingBytes + 1024 /*align*/ + 256 /*barriers*/;

// Vocab columns per forward statistics partial (= the GEMM's N tile).
constexpr int kVTile = kBN;
// Rows per block of the merge kernel (one merge block partial per 32 rows).
constexpr int kMergeRows = 32;

// Workspace header (offset 0 of every workspace).
struct Header {
  int32_t status;    // FLCE_ERR_LABEL | FLCE_ERR_TIMEOUT | FLCE_ERR_NONFINITE bits
  uint32_t ticket;   // last-block election in the merge kernel
  int64_t n_valid;   // rows whose label is not ignore_index
  double loss_sum;   // sum of row losses over finished chunks (fixed order)
  int64_t correct;   // valid rows whose argmax equals the label
};

enum KernelId {
  K_PROLOGUE = 0,
  K_FWD_GEMM = 1,
  K_MERGE = 2,
  K_DLOGITS = 3,
  K_GRADH_GEMM = 4,
  K_GRADW_GEMM = 5,
  K_TRANSPOSE_W = 6,
  K_TRANSPOSE_H = 7,
  K_FINISH = 8,
  K_SIMT_STATS = 9,
  K_CE_STATS = 10,
  K_CE_GRAD = 11,
  K_RECOMPUTE_GEMM = 12,
  K_CONVERT = 13,
  K_SCALE = 14,
  K_VP_MERGE = 15,
  K_SPLIT = 16,
};

enum EpiMode {
  EPI_STATS = 0,        // forward statistics partials only
  EPI_STATS_STORE = 1,  // statistics partials + capped logits s stored (fp32)
  EPI_BF16 = 2,         // out = bf16(alpha * acc)
  EPI_ACC_F32 = 3,      // out += alpha * acc (fp32)
  EPI_DZ = 4,           // out = bf16 dlogits formed from z = alpha * acc, lse and labels
  EPI_F32 = 5,          // out = alpha * acc (fp32, bulk store)
  EPI_STATS_STORE16 = 6,  // statistics partials + s stored as fp16 s - gmax, gmax (fp32) per 32 columns
};

struct GemmParams {
  // D [M, N] = A [M, K] * B [N, K]^T, both operands K-major bf16.
  int M, N, K;
  int m_tiles, n_tiles, k_iters, group_m;
  int a_row0, b_row0;  // row offsets added to the TMA row coordinates
  float alpha;
  int M_valid;  // rows of D that are written
  int N_valid;  // columns of D that are valid
  // statistics epilogue
  float softcap, inv_softcap;
  const int64_t* labels;  // labels of D's rows (already offset to row 0 of D)
  int64_t ignore_index;
  float* part_max;  // [n_tiles][ldp]
  float* part_sum;  // [n_tiles][ldp]
  int32_t* part_idx;  // [n_tiles][ldp]
  // 1: the call returns no predicted tokens, so part_idx carries only what the
  // token accuracy needs (the label's column where the label is the tile's
  // first maximum, else another column of the tile) and the epilogue skips
  // the argmax; 0 (the default): part_idx is the tile's first maximum
  int no_argmax;
  float* tgt;       // [ldp]  capped logit at the label
  int ldp;
  float* zbuf;  // capped logits [rows][ldz] (STATS_STORE, and the SIMT path)
  int64_t ldz;
  float* gmax;  // STATS_STORE16: [rows][ldg] maximum of each 32-column group of s
  int64_t ldg;
  // plain epilogues
  void* out;
  int64_t ldo;
  // Column j of D is vocab index col0 + j: the statistics epilogues compare
  // labels (global vocab ids) with it, and EPI_DZ places the one-hot term by
  // it (0 unless D covers a vocab slab or a vocab shard).
  // dlogits epilogue (EPI_DZ):
  const float* lse;  // [rows of D]
  const struct Header* hdr;
  float grad_scale;
  int reduction;
  int col0;
  // 1: the epilogue's bulk stores / reduce-adds (EPI_STATS_STORE, EPI_F32,
  // EPI_ACC_F32) carry an L2 evict-first policy; the engine sets it for the
  // stored logits only (on the fp32 accumulators it measured no faster)
  int store_hint;
  // control
  int32_t* status;
  uint64_t timeout_ns;
  int debug_flags;
};

// Tensor-core GEMM (tcgen05 + TMA + TMEM), persistent over `grid` CTAs.
// a_mn / b_mn: the operand is MN-major in global memory ([K rows][MN cols]),
// loaded as 64x64 boxes; otherwise K-major ([MN rows][K cols]).
// c: fp32 output tensor map with 32 x 32 boxes and 128-byte swizzle, used by
// EPI_STATS_STORE (the stored logits, bulk store) and EPI_ACC_F32 (bulk
// reduce-add into the fp32 accumulator); ignored by the other modes.
// wide: 256 x 256 CTA tiles (two M = 128 MMAs per K step sharing the B slice,
// one 512-column accumulator) instead of 128 x 256 tiles with two accumulators;
// the all-K-major backward combinations always use 128-row tiles. grid is the
// largest number of CTAs to launch (at most one per tile).
// pair (with wide): the 256 x 256 tile is computed by a cluster of two CTAs on
// two SMs with tcgen05 cta_group::2 (M = 256): each CTA loads 128 rows of A
// and 128 of the 256 rows of B, and keeps its 128 rows of the tile in two
// 256-column TMEM accumulators, so the epilogue overlaps the next tile's MMAs.
// A K-major B operand then needs a tensor map with 128-row boxes.
cudaError_t launch_gemm_tc(int mode, bool a_mn, bool b_mn, bool wide, const CUtensorMap* a, const CUtensorMap* b,
                           const CUtensorMap* c, const GemmParams& p, int grid, cudaStream_t s, bool pair = false);
// The same GEMM on fp32 operands (tcgen05 kind::tf32), both K-major; modes
// EPI_STATS, EPI_STATS_STORE, EPI_F32, EPI_ACC_F32.
// a_lo / b_lo (both or neither): the three-pass split for fp32 accuracy; a and
// b then hold hi = tf32(x), a_lo and b_lo lo = x - hi (128-row tiles).
cudaError_t launch_gemm_tc_tf32(int mode, bool wide, const CUtensorMap* a, const CUtensorMap* b,
                                const CUtensorMap* c, const GemmParams& p, int grid, cudaStream_t s,
                                const CUtensorMap* a_lo = nullptr, const CUtensorMap* b_lo = nullptr);
// Debug GEMM on the fp32 FMA pipes; writes alpha*acc to zbuf for the statistics
// modes (then run launch_stats_from_z) and behaves like the tensor-core GEMM
// for the plain modes.
cudaError_t launch_gemm_simt(int mode, const void* A, int64_t lda, const void* B, int64_t ldb,
                             const GemmParams& p, cudaStream_t s);
cudaError_t launch_stats_from_z(const GemmParams& p, int rows, bool store, cudaStream_t s);

cudaError_t launch_prologue(const int64_t* labels, int64_t n, int64_t vocab, int64_t ignore_index,
                            Header* hdr, cudaStream_t s);
struct MergeParams {
  int rows;            // rows in this chunk
  int n_vtiles;
  int ldp;
  const float* part_max;
  const float* part_sum;
  const int32_t* part_idx;
  const float* tgt;
  const int64_t* labels;  // chunk labels
  int64_t ignore_index;
  float* lse;             // [rows] chunk workspace
  int64_t* predicted;     // global output offset to the chunk, or null
  float* row_lse;         // global output offset to the chunk, or null
  float* row_loss;        // global output offset to the chunk, or null (0 on ignored rows)
  double* block_loss;     // [blocks]
  int64_t* block_correct; // [blocks]
  Header* hdr;
  // Vocab shard (flce_vp_forward): when shard_out is set, the merge writes the
  // shard's per-row partials instead of lse / loss / predictions: shard_out +
  // f * ld_shard + row for fields f = max, sum of exp, argmax (int32 global id
  // in the float word: vocab_offset + the tile index), label logit (0 when the
  // label is outside [vocab_offset, vocab_offset + vocab_shard)).
  float* shard_out;
  int64_t ld_shard;
  int64_t vocab_offset;
  int64_t vocab_shard;
};
cudaError_t launch_merge(const MergeParams& p, cudaStream_t s);

// Merge of the per-row partials of S vocab shards (flce_vp_backward), in
// shard order: lse, argmax (lowest global id on ties), the label's logit from
// the shard that holds the label, the row loss, and the fixed-order batch sums.
constexpr int kMaxShards = 64;
struct VpMergeParams {
  int rows;                      // N
  int n_shards;                  // S <= kMaxShards
  int32_t offsets[kMaxShards + 1];  // vocab offset of each shard, then vocab_total
  const float* partials;         // [S][4][ld]
  int64_t ld;
  const int64_t* labels;
  int64_t ignore_index;
  float* lse;                    // [rows] (workspace)
  int64_t* predicted;            // [rows] or null
  float* row_lse;                // [rows] or null
  double* block_loss;            // [ceil(rows / 32)]
  int64_t* block_correct;
  Header* hdr;
};
cudaError_t launch_vp_merge(const VpMergeParams& p, cudaStream_t s);

struct DlogitParams {
  int rows, vocab;
  const float* s;   // capped logits [rows][lds]
  int64_t lds;
  const uint16_t* s16;  // or: fp16 s - gmax [rows][lds] (the bf16 product path)
  const float* gmax;    // with s16: [rows][ldg], the reference of each 32-column group
  int64_t ldg;
  const float* lse; // [rows]
  const int64_t* labels;
  int64_t label_offset;  // vocab id of column 0 (a vocab shard's offset; 0 otherwise)
  int64_t ignore_index;
  float softcap, inv_softcap;
  float grad_scale;
  int reduction;
  const Header* hdr;
  uint16_t* dz;     // bf16 [rows][ldd] or null
  int64_t ldd;
  uint16_t* dzt;    // bf16 [vocab][ldt] or null
  int64_t ldt;
  float* dz32;      // fp32-operand path: dz [rows][ldd] and dz^T [vocab][ldt] in fp32
  float* dzt32;
  float* dz32_lo;   // three-pass tf32: dz32 / dzt32 then get tf32(dz), these dz - tf32(dz)
  float* dzt32_lo;
};
cudaError_t launch_dlogits(const DlogitParams& p, cudaStream_t s);

// out [cols][ldo] = in [rows][ldi]^T, bf16 / fp32.
cudaError_t launch_transpose_bf16(const uint16_t* in, int64_t ldi, int rows, int cols, uint16_t* out,
                                  int64_t ldo, cudaStream_t s);
// out_lo non-null: out receives tf32(x) and out_lo x - tf32(x) (the split).
cudaError_t launch_transpose_f32(const float* in, int64_t ldi, int rows, int cols, float* out, int64_t ldo,
                                 cudaStream_t s, float* out_lo = nullptr);
// hi / lo [rows][ldo] = the tf32 split of in [rows][ldi] (cols columns).
cudaError_t launch_split_f32(const float* in, int64_t ldi, int rows, int cols, float* hi, float* lo, int64_t ldo,
                             cudaStream_t s);

// Columns per warp task of the cross-entropy-on-logits statistics.
constexpr int kCeTile = 8192;

struct CeParams {
  int rows, vocab, n_vtiles, ldp;
  int dtype;          // FLCE_DTYPE_*
  int vec_ok;         // rows are 16-byte aligned: vector loads / stores
  const void* logits;
  int64_t ldx;
  void* grad;
  int64_t ldg;
  const int64_t* labels;
  int64_t ignore_index;
  float out_mult, softcap, inv_softcap, grad_scale;
  int reduction;
  const float* row_scale;
  float* part_max;
  float* part_sum;
  int32_t* part_idx;
  float* tgt;
  const float* lse;
  const Header* hdr;
};
cudaError_t launch_ce_stats(const CeParams& p, cudaStream_t s);
cudaError_t launch_ce_grad(const CeParams& p, cudaStream_t s);

// out [n] (bf16) = in [n] (fp32), round to nearest even.
cudaError_t launch_f32_to_bf16(const float* in, uint16_t* out, int64_t n, cudaStream_t s);

// y [n] = scale * x [n], converted (bf16 results rounded to nearest even);
// scale is a device float or nullptr for 1. x == y only when the types match.
cudaError_t launch_scale_convert(const void* x, bool x_f32, void* y, bool y_f32, int64_t n, const float* scale,
                                 int sms, cudaStream_t s);

cudaError_t launch_finish(const Header* hdr, int reduction, float* loss, float* token_accuracy,
                          cudaStream_t s);

}  // namespace flce
