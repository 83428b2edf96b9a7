// Persistent tcgen05 GEMM with fused epilogues: D [M, N] = A [M, K] * B [N, K]^T.
//
// One CTA per SM, warp-specialised, in two tile shapes (template TMH):
//   warp 0      one lane issues TMA loads of the A and B slices of each 64-deep
//               K step into a shared-memory ring (128-byte swizzle);
//   warp 1      owns the 512 TMEM columns; one lane issues tcgen05.mma
//               (M=128, N=256, K=16 per instruction, fp32 accumulate);
//   warps 2..   the epilogue: the thread on TMEM lane r owns row r of a 128-row
//               half of the tile, reads 32 columns at a time with tcgen05.ld
//               and applies the mode's epilogue.
// TMH = 1: 128 x 256 tiles, 192 threads, a 4-stage ring of 48 KB stages and two
//   256-column accumulators, so the epilogue of tile t overlaps the main loop
//   of tile t+1 (four epilogue warps).
// TMH = 2: 256 x 256 tiles, 320 threads, a 3-stage ring of 64 KB stages; two
//   MMAs per K step (one per 128-row half of A) share the B slice, which takes
//   a third less operand traffic into the SM per flop; the single 512-column
//   accumulator is drained by eight epilogue warps.
// Epilogue modes: forward statistics of the linear cross-entropy (softcap,
// running max / sum of exponentials, argmax, label logit) with or without
// storing the capped logits (fp32, or fp16 relative to each 32-column group's
// maximum); bf16 store of alpha*acc (grad_h); fp32 accumulate-in-place of
// alpha*acc (grad_W += ...); bf16 dlogits from recomputed logits (EPI_DZ).
// A CTA-pair variant (gemm_tc_pair_kernel, below) computes 256 x 256 tiles on
// two SMs with cta_group::2, and a three-pass split (SPLIT) gives fp32
// operands fp32 accuracy on the tf32 tensor cores.
// Every wait is bounded (FLCE_ERR_TIMEOUT); on the way out the CTA drains the
// copies and MMAs it issued and frees TMEM.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include <atomic>

#include "flce_device.cuh"
#include "flce_epilogue.cuh"

namespace flce {

// Grouped rasterisation: tiles walk group_m row-tiles at a time, row-tile
// fastest, so the CTAs resident at once share a few B slices and a few A
// slices in L2.
// Tile t of the walk: groups of `group` M-units, M fastest within a group. An
// M-unit is TMH consecutive 128-row tiles (one CTA tile of TMH * 128 rows).
__device__ __forceinline__ void tile_coords(const GemmParams& p, int units_m, int group, int t, int& mu, int& nb) {
  const int per_group = group * p.n_tiles;
  const int g = t / per_group;
  const int first_m = g * group;
  const int gsize = min(units_m - first_m, group);
  const int local = t - g * per_group;
  mu = first_m + local % gsize;
  nb = local / gsize;
}

// Staging of one epilogue warp's 32 x 32 fp32 sub-tile for a TMA bulk store or
// reduce-add: lane r writes its row as eight 16-byte chunks, chunk q at slot
// q ^ (r & 7) (the 128-byte swizzle the tensor map expects; also spreads the
// writes of a warp over all banks). With two buffers they alternate and lane 0
// keeps at most one older copy reading shared memory; with one, lane 0 waits
// for the previous copy's reads before the buffer is rewritten.
struct EpiStage {
  uint8_t* base;    // this warp's buffers
  int next;         // buffer to fill next
  int nbuf;         // 1 or 2
  uint64_t policy;  // L2 policy of the global writes (when hint)
  bool hint;
};

// Walks the 256 accumulator columns of this thread's row in chunks of 32,
// calling f(r, c) for chunk c, with the TMEM load of chunk c + 1 in flight
// while chunk c is processed (two register buffers).
template <typename F>
__device__ __forceinline__ void tmem_row_chunks(uint32_t tcol, F&& f) {
  uint32_t ra[32], rb[32];
  tmem_load_32cols(tcol, ra);
#pragma unroll 1
  for (int c = 0; c < kBN / 32; c += 2) {
    tmem_load_wait_regs(ra);
    tmem_load_32cols(tcol + (c + 1) * 32, rb);
    f(ra, c);
    tmem_load_wait_regs(rb);
    if (c + 2 < kBN / 32) tmem_load_32cols(tcol + (c + 2) * 32, ra);
    f(rb, c + 1);
  }
}

template <bool REDUCE>
__device__ __forceinline__ void stage_and_send(EpiStage& es, const CUtensorMap* map, int lane, const float (&v)[32],
                                               int32_t x, int32_t y) {
  uint8_t* buf = es.base + es.next * kStageBufBytes;
  if (lane == 0) {  // the copy that last used `buf` has read it
    if (es.nbuf == 2)
      bulk_wait_group_read<1>();
    else
      bulk_wait_group_read<0>();
  }
  __syncwarp();
  float4* row = reinterpret_cast<float4*>(buf + lane * 128);
#pragma unroll
  for (int q = 0; q < 8; ++q) row[q ^ (lane & 7)] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    if (es.hint) {
      if (REDUCE)
        tma_reduce_add_2d_hint(map, buf, x, y, es.policy);
      else
        tma_store_2d_hint(map, buf, x, y, es.policy);
    } else {
      if (REDUCE)
        tma_reduce_add_2d(map, buf, x, y);
      else
        tma_store_2d(map, buf, x, y);
    }
    bulk_commit_group();
  }
  if (es.nbuf == 2) es.next ^= 1;
}

// The same staging for two 32-column groups of fp16 values (a 32 x 64 fp16
// sub-tile, again 128 bytes per row): lo holds columns x .. x+31, hi the next 32.
__device__ __forceinline__ void stage_and_send16(EpiStage& es, const CUtensorMap* map, int lane,
                                                 const uint32_t (&lo)[16], const uint32_t (&hi)[16], int32_t x,
                                                 int32_t y) {
  uint8_t* buf = es.base + es.next * kStageBufBytes;
  if (lane == 0) {
    if (es.nbuf == 2)
      bulk_wait_group_read<1>();
    else
      bulk_wait_group_read<0>();
  }
  __syncwarp();
  uint4* row = reinterpret_cast<uint4*>(buf + lane * 128);
#pragma unroll
  for (int q = 0; q < 4; ++q) row[q ^ (lane & 7)] = make_uint4(lo[4 * q], lo[4 * q + 1], lo[4 * q + 2], lo[4 * q + 3]);
#pragma unroll
  for (int q = 0; q < 4; ++q)
    row[(q + 4) ^ (lane & 7)] = make_uint4(hi[4 * q], hi[4 * q + 1], hi[4 * q + 2], hi[4 * q + 3]);
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    if (es.hint)
      tma_store_2d_hint(map, buf, x, y, es.policy);
    else
      tma_store_2d(map, buf, x, y);
    bulk_commit_group();
  }
  if (es.nbuf == 2) es.next ^= 1;
}

__device__ __forceinline__ uint32_t pack_half2(float a, float b) {
  const __half2 v = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// Forward statistics of one 256-column tile of 128 rows. STORE: 0 keeps only
// the statistics; 1 also stores the capped logits s in fp32; 2 stores them
// relative to the maximum of their 32-column group, s - gmax, in fp16 (halving
// the stored bytes), with gmax in fp32 beside them.
// ARGMAX: the partial index is the tile's first maximum; without it (calls that
// need the token accuracy but not the predicted tokens) the index is the
// label's column when the label is the tile's first maximum, and otherwise a
// column of the tile other than the label's. The merge then takes the index of
// the first tile that holds the row's maximum, as before, and it equals the
// label exactly when the label is the row's first maximum.
template <int STORE, bool ARGMAX>
__device__ __forceinline__ void epilogue_stats(const GemmParams& p, const CUtensorMap* zmap, EpiStage& es,
                                               uint32_t tcol, int mb, int nb, int quarter, int lane) {
  const int row = quarter * 32 + lane;
  const int grow = mb * kBM + row;
  const bool row_ok = grow < p.M_valid;
  const int64_t label = row_ok ? __ldg(p.labels + grow) : p.ignore_index;
  const int n0 = nb * kBN;
  const int64_t ylocal = label - p.col0;  // the label as a column of D
  const bool has_label = label != p.ignore_index && ylocal >= n0 && ylocal < n0 + kBN;
  const bool full_tile = n0 + kBN <= p.N_valid;  // no column past V: skip the mask
  const int ycol = has_label ? static_cast<int>(ylocal) : -1;  // the label's column in this tile, or -1
  RowStats st;
  row_stats_init(st, n0);
  uint32_t held[16];  // STORE == 2: the even group's fp16 values, sent with the odd one
  float gm0 = 0.f, gm1 = 0.f, gm2 = 0.f;  // STORE == 2: gmax of groups 4k .. 4k+2, stored with 4k+3
  tmem_row_chunks(tcol, [&](const uint32_t(&r)[32], int c) {
    float s[32];
    const int col0 = n0 + c * 32;
    if (p.softcap > 0.f) {
      softcap32(s, r, p.alpha, p.softcap, p.inv_softcap);
    } else if (p.alpha != 1.f) {
      const uint64_t al2 = f2_pack(p.alpha, p.alpha);
#pragma unroll
      for (int j = 0; j < 32; j += 2)
        f2_unpack(f2_mul(f2_pack(__uint_as_float(r[j]), __uint_as_float(r[j + 1])), al2), s[j], s[j + 1]);
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) s[j] = __uint_as_float(r[j]);
    }
    if (!full_tile) {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (col0 + j >= p.N_valid) s[j] = -INFINITY;
    }
    if (STORE == 1) stage_and_send<false>(es, zmap, lane, s, col0, mb * kBM + quarter * 32);
    const float cm = ARGMAX ? row_stats_update32(st, s, col0, ycol) : row_stats_update32_noarg(st, s, ycol - col0);
    if (STORE == 2) {
      // A group wholly past V has cm = -inf: its values are stored as -inf
      // (never read) and its gmax as 0.
      const float ref = cm == -INFINITY ? 0.f : cm;
      const uint64_t nref2 = f2_pack(-ref, -ref);
      uint32_t hv[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        float d0, d1;
        f2_unpack(f2_add(f2_pack(s[2 * j], s[2 * j + 1]), nref2), d0, d1);
        hv[j] = pack_half2(d0, d1);
      }
      // four groups' maxima in one 16-byte store (ldg and the tile's first
      // group are multiples of 8)
      const int q = c & 3;
      if (q == 0) {
        gm0 = ref;
      } else if (q == 1) {
        gm1 = ref;
      } else if (q == 2) {
        gm2 = ref;
      } else if (row_ok) {
        *reinterpret_cast<float4*>(p.gmax + static_cast<int64_t>(grow) * p.ldg + (col0 >> 5) - 3) =
            make_float4(gm0, gm1, gm2, ref);
      }
      if ((c & 1) == 0) {
#pragma unroll
        for (int j = 0; j < 16; ++j) held[j] = hv[j];
      } else {
        stage_and_send16(es, zmap, lane, held, hv, col0 - 32, mb * kBM + quarter * 32);
      }
    }
  });
  if (row_ok) {
    const int64_t o = static_cast<int64_t>(nb) * p.ldp + grow;
    p.part_max[o] = st.mx;
    p.part_sum[o] = st.sum;
    if (ARGMAX)
      p.part_idx[o] = st.arg;
    else
      p.part_idx[o] = (has_label && st.first && st.tgt == st.mx) ? ycol : (ycol == n0 ? n0 + 1 : n0);
    if (has_label) p.tgt[grow] = st.tgt;
  }
}

// The statistics epilogue in the form the call asks for (GemmParams::no_argmax).
template <int STORE>
__device__ __forceinline__ void epilogue_stats_any(const GemmParams& p, const CUtensorMap* zmap, EpiStage& es,
                                                   uint32_t tcol, int mb, int nb, int quarter, int lane) {
  if (p.no_argmax)
    epilogue_stats<STORE, false>(p, zmap, es, tcol, mb, nb, quarter, lane);
  else
    epilogue_stats<STORE, true>(p, zmap, es, tcol, mb, nb, quarter, lane);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ void epilogue_bf16(const GemmParams& p, uint32_t tcol, int mb, int nb, int row) {
  const int grow = mb * kBM + row;
  const bool row_ok = grow < p.M_valid;
  const int n0 = nb * kBN;
  uint16_t* orow = static_cast<uint16_t*>(p.out) + static_cast<int64_t>(grow) * p.ldo + n0;
  tmem_row_chunks(tcol, [&](const uint32_t(&r)[32], int c) {
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const int col = n0 + c * 32 + g * 8;
      if (row_ok && col < p.N_valid) {
        uint4 v;
        v.x = pack_bf16x2(__uint_as_float(r[g * 8 + 0]) * p.alpha, __uint_as_float(r[g * 8 + 1]) * p.alpha);
        v.y = pack_bf16x2(__uint_as_float(r[g * 8 + 2]) * p.alpha, __uint_as_float(r[g * 8 + 3]) * p.alpha);
        v.z = pack_bf16x2(__uint_as_float(r[g * 8 + 4]) * p.alpha, __uint_as_float(r[g * 8 + 5]) * p.alpha);
        v.w = pack_bf16x2(__uint_as_float(r[g * 8 + 6]) * p.alpha, __uint_as_float(r[g * 8 + 7]) * p.alpha);
        *reinterpret_cast<uint4*>(orow + c * 32 + g * 8) = v;
      }
    }
  });
}

// grad_W (or the recompute path's fp32 grad_h) += alpha * acc: the sub-tile is
// staged in shared memory and added in L2 by a TMA bulk reduce-add; rows and
// columns outside the tensor map are clipped by the copy engine.
template <bool REDUCE>
__device__ __forceinline__ void epilogue_out_f32(const GemmParams& p, const CUtensorMap* omap, EpiStage& es,
                                                 uint32_t tcol, int mb, int nb, int quarter, int lane) {
  const int n0 = nb * kBN;
  tmem_row_chunks(tcol, [&](const uint32_t(&r)[32], int c) {
    float v[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]) * p.alpha;
    if (n0 + c * 32 < p.N_valid) stage_and_send<REDUCE>(es, omap, lane, v, n0 + c * 32, mb * kBM + quarter * 32);
  });
}

// Recompute pass of the low-memory backward: z = alpha * acc is capped, turned
// into dlogits with the row's lse and label, rounded to bf16 and stored.
__device__ __forceinline__ void epilogue_dz(const GemmParams& p, uint32_t tcol, int mb, int nb, int row,
                                            float coef) {
  const int grow = mb * kBM + row;
  const bool row_ok = grow < p.M_valid;
  const int64_t label = row_ok ? __ldg(p.labels + grow) : p.ignore_index;
  const bool valid = row_ok && label != p.ignore_index;
  const float ci = valid ? coef : 0.f;
  const float lse = row_ok ? __ldg(p.lse + grow) : 0.f;
  const int n0 = nb * kBN;
  const int64_t ylocal = valid ? label - p.col0 : -1;
  uint16_t* orow = static_cast<uint16_t*>(p.out) + static_cast<int64_t>(grow) * p.ldo + n0;
#pragma unroll 1
  for (int c = 0; c < kBN / 32; ++c) {
    uint32_t r[32];
    tmem_load_32cols(tcol + c * 32, r);
    tmem_load_wait();
    float sv[32];  // the capped logits, as the forward statistics computed them
    if (p.softcap > 0.f) {
      softcap32(sv, r, p.alpha, p.softcap, p.inv_softcap);
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) sv[j] = __uint_as_float(r[j]) * p.alpha;
    }
    float d[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      float q = __expf(sv[j] - lse) - (static_cast<int64_t>(n0 + c * 32 + j) == ylocal ? 1.f : 0.f);
      if (p.softcap > 0.f) {
        const float u = sv[j] * p.inv_softcap;
        q *= (1.f - u * u);
      }
      d[j] = ci * q;
    }
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const int col = n0 + c * 32 + g * 8;
      if (row_ok && col < p.N_valid) {
        uint4 v;
        v.x = pack_bf16x2(d[g * 8 + 0], d[g * 8 + 1]);
        v.y = pack_bf16x2(d[g * 8 + 2], d[g * 8 + 3]);
        v.z = pack_bf16x2(d[g * 8 + 4], d[g * 8 + 5]);
        v.w = pack_bf16x2(d[g * 8 + 6], d[g * 8 + 7]);
        *reinterpret_cast<uint4*>(orow + c * 32 + g * 8) = v;
      }
    }
  }
}

// TF32: operands are fp32 (read by the tensor cores as tf32); a K slice is then
// 32 elements, still one 128-byte swizzle row, and one MMA covers K = 8.
// TMH = 1: 128 x 256 CTA tiles, a 4-stage ring and two 256-column TMEM
// accumulators (the epilogue of one tile overlaps the MMAs of the next).
// TMH = 2: 256 x 256 CTA tiles as two M = 128 MMAs sharing each B slice, a
// 3-stage ring of the same size and one 512-column accumulator: a third less
// operand traffic into the SM per flop. The accumulator is drained by eight
// epilogue warps, two per TMEM lane quarter (warps 2-5 rows 0-127, warps 6-9
// rows 128-255, one staging buffer each), so the tensor cores wait for half
// as long between tiles as four warps would make them.
// SPLIT (tf32 only, 128-row tiles): three-pass tf32 for fp32 accuracy. Each
// fp32 operand comes as two arrays, hi = x rounded to tf32 and lo = x - hi
// (tma_a / tma_b and tma_a2 / tma_b2), and every K step issues
// hi*hi + hi*lo + lo*hi into the same accumulator; the dropped lo*lo term
// and the tf32 rounding of lo are about 2^-21 of each product. A stage then
// holds both halves of A and B (96 KB), so the ring has two stages.
template <int MODE, bool A_MN, bool B_MN, bool TF32, int TMH, bool SPLIT = false>
__global__ void __launch_bounds__(gemm_threads(TMH), 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tma_a, const __grid_constant__ CUtensorMap tma_b,
                   const __grid_constant__ CUtensorMap tma_c, const __grid_constant__ CUtensorMap tma_a2,
                   const __grid_constant__ CUtensorMap tma_b2, const GemmParams p) {
  static_assert(!SPLIT || (TF32 && TMH == 1), "the three-pass split is for tf32 on 128-row tiles");
  constexpr int S = SPLIT ? 2 : TMH == 2 ? 3 : kStages;
  constexpr int AHalf = kAStageBytes * TMH;          // one copy of A's slice
  constexpr int ABytes = AHalf * (SPLIT ? 2 : 1);    // hi then lo
  constexpr int BBytes = kBStageBytes * (SPLIT ? 2 : 1);
  constexpr int NBUF = TMH == 2 ? 1 : 2;
  static_assert(S * (ABytes + BBytes) <= kStages * (kAStageBytes + kBStageBytes), "ring exceeds the budget");
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  uint8_t* sA = smem;
  uint8_t* sB = smem + S * ABytes;
  uint8_t* sStage = smem + kStages * (kAStageBytes + kBStageBytes);  // epilogue staging, 32 KB
  uint64_t* full = reinterpret_cast<uint64_t*>(sStage + kEpiStagingBytes);
  uint64_t* empty = full + S;
  uint64_t* tfull = empty + S;
  uint64_t* tempty = tfull + 2;
  uint64_t* mma_done = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

  static_assert(!(TF32 && (A_MN || B_MN)), "tf32 operands are K-major only");
  constexpr int kSliceK = TF32 ? kBK / 2 : kBK;  // elements per 128-byte K slice
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], TMH == 2 ? 256 : 128);  // every epilogue thread arrives
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tma_a);
    tma_prefetch_desc(&tma_b);
    if (MODE == EPI_STATS_STORE || MODE == EPI_STATS_STORE16 || MODE == EPI_ACC_F32 || MODE == EPI_F32)
      tma_prefetch_desc(&tma_c);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;

  const WaitCtx wc{abort_flag, p.status, p.timeout_ns};
  const int units_m = (p.m_tiles + TMH - 1) / TMH;
  const int group = p.group_m / TMH > 0 ? p.group_m / TMH : 1;
  const int total = units_m * p.n_tiles;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      bool aborted = false;
      if (!(p.debug_flags & FLCE_FLAG_TEST_STALL)) {
        for (int t = blockIdx.x; t < total && !aborted; t += gridDim.x) {
          int mu, nb;
          tile_coords(p, units_m, group, t, mu, nb);
          const int row0 = p.a_row0 + mu * kBM * TMH;
          for (int k = 0; k < p.k_iters; ++k) {
            if (!wait_bounded(&empty[stage], phase ^ 1u, wc)) {
              aborted = true;
              break;
            }
            mbar_arrive_expect_tx(&full[stage], ABytes + BBytes);
            // K-major operand: boxes of 64 K x 128 (A) or 256 (B) rows.
            // MN-major operand: boxes of 64 MN x 64 K, one per 64 rows of the
            // tile, 8 KB apart.
            if (A_MN) {
#pragma unroll
              for (int j = 0; j < kBM * TMH / 64; ++j)
                tma_load_2d(sA + stage * ABytes + j * 8192, &tma_a, &full[stage], row0 + j * 64, k * kSliceK);
            } else {
#pragma unroll
              for (int hh = 0; hh < TMH; ++hh)
                tma_load_2d(sA + stage * ABytes + hh * kAStageBytes, &tma_a, &full[stage], k * kSliceK,
                            row0 + hh * kBM);
            }
            if (B_MN) {
#pragma unroll
              for (int j = 0; j < kBN / 64; ++j)
                tma_load_2d(sB + stage * BBytes + j * 8192, &tma_b, &full[stage], p.b_row0 + nb * kBN + j * 64,
                            k * kSliceK);
            } else {
              tma_load_2d(sB + stage * BBytes, &tma_b, &full[stage], k * kSliceK, p.b_row0 + nb * kBN);
            }
            if (SPLIT) {
              tma_load_2d(sA + stage * ABytes + AHalf, &tma_a2, &full[stage], k * kSliceK, row0);
              tma_load_2d(sB + stage * BBytes + kBStageBytes, &tma_b2, &full[stage], k * kSliceK,
                          p.b_row0 + nb * kBN);
            }
            ++issued;
            if (++stage == S) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      if (aborted) {
        // The most recent min(issued, S) loads may still be in flight:
        // wait for each to land before this CTA's shared memory goes away.
        const int n = issued < S ? issued : S;
        int s = stage;
        uint32_t ph = phase;
        for (int i = 0; i < n; ++i) {
          if (s == 0) {
            s = S - 1;
            ph ^= 1u;
          } else {
            --s;
          }
          wait_drain(&full[s], ph, p.timeout_ns, p.status);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool aborted = false;
      constexpr uint32_t idesc = TF32 ? idesc_tf32_f32(kBM, kBN) : idesc_bf16_f32(kBM, kBN, A_MN, B_MN);
      const uint32_t a_base = smem_u32(sA);
      const uint32_t b_base = smem_u32(sB);
      for (int t = blockIdx.x; t < total && !aborted; t += gridDim.x) {
        if (!wait_bounded(&tempty[acc], acc_phase ^ 1u, wc)) break;
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kBN);
        for (int k = 0; k < p.k_iters; ++k) {
          if (!wait_bounded(&full[stage], phase, wc)) {
            aborted = true;
            break;
          }
          tc_fence_after_sync();
          const uint32_t a0 = a_base + stage * ABytes;
          const uint32_t b0 = b_base + stage * BBytes;
          if (SPLIT) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t ah = sdesc_kmajor_sw128(a0 + kk * 32);
              const uint64_t al = sdesc_kmajor_sw128(a0 + AHalf + kk * 32);
              const uint64_t bh = sdesc_kmajor_sw128(b0 + kk * 32);
              const uint64_t bl = sdesc_kmajor_sw128(b0 + kBStageBytes + kk * 32);
              tc_mma_tf32(d_tmem, ah, bh, idesc, (k | kk) != 0 ? 1u : 0u);
              tc_mma_tf32(d_tmem, ah, bl, idesc, 1u);
              tc_mma_tf32(d_tmem, al, bh, idesc, 1u);
            }
          }
#pragma unroll
          for (int kk = 0; kk < (SPLIT ? 0 : 4); ++kk) {
            // One MMA per 32 B of K (16 bf16 or 8 tf32 elements): 32 B along a
            // K-major row, or two 8-row K groups (2048 B) of an MN-major tile.
            // With TMH = 2 the second M half of A starts 16 KB further on (128
            // K-major rows, or two 64-wide MN blocks) and accumulates into
            // TMEM columns 256-511.
            const uint64_t bd = B_MN ? sdesc_mnmajor_sw128(b0 + kk * 2048) : sdesc_kmajor_sw128(b0 + kk * 32);
#pragma unroll
            for (int hh = 0; hh < TMH; ++hh) {
              const uint32_t ah = a0 + hh * kAStageBytes;
              const uint64_t ad = A_MN ? sdesc_mnmajor_sw128(ah + kk * 2048) : sdesc_kmajor_sw128(ah + kk * 32);
              if (TF32)
                tc_mma_tf32(d_tmem + hh * kBN, ad, bd, idesc, (k | kk) != 0 ? 1u : 0u);
              else
                tc_mma_bf16(d_tmem + hh * kBN, ad, bd, idesc, (k | kk) != 0 ? 1u : 0u);
            }
          }
          tc_commit(&empty[stage]);
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (aborted) break;
        tc_commit(&tfull[acc]);
        if (NBUF == 2) {
          acc ^= 1;
          if (acc == 0) acc_phase ^= 1u;
        } else {
          acc_phase ^= 1u;
        }
      }
      // All issued tensor-core work must finish before TMEM is released.
      tc_commit(mma_done);
      wait_drain(mma_done, 0, p.timeout_ns, p.status);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    float coef = 0.f;  // dlogits scale c of the EPI_DZ epilogue
    if (MODE == EPI_DZ) {
      const int64_t nv = p.hdr->n_valid;
      if (nv > 0) coef = p.reduction == FLCE_REDUCTION_MEAN ? p.grad_scale / static_cast<float>(nv) : p.grad_scale;
    }
    const int quarter = warp & 3;  // TMEM lanes this warp may access
    const int row = quarter * 32 + lane;
    const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
    // TMH = 1: four warps, two 4 KB buffers each, all of the tile's rows.
    // TMH = 2: eight warps, one buffer each; warp 2 + 4 * half + q drains the
    // 128-row half `half` of the 256-row tile.
    const int half = TMH == 2 ? (warp - 2) / 4 : 0;
    EpiStage es{sStage + (warp - 2) * (TMH == 2 ? 1 : 2) * kStageBufBytes, 0, TMH == 2 ? 1 : 2, 0,
                p.store_hint != 0};
    if (es.hint) es.policy = l2_policy_evict_first();
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      int mu, nb;
      tile_coords(p, units_m, group, t, mu, nb);
      bool ok = wait_bounded(&tfull[acc], acc_phase, wc);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after_sync();
#pragma unroll 1
      for (int hh = half; hh < half + 1; ++hh) {
        // 128-row tile mb of the output, held in TMEM columns tcol..tcol+255
        const int mb = mu * TMH + hh;
        if (mb >= p.m_tiles) break;
        const uint32_t tcol = t_lane + static_cast<uint32_t>((acc + hh) * kBN);
        if (MODE == EPI_STATS) {
          epilogue_stats_any<0>(p, &tma_c, es, tcol, mb, nb, quarter, lane);
        } else if (MODE == EPI_STATS_STORE) {
          epilogue_stats_any<1>(p, &tma_c, es, tcol, mb, nb, quarter, lane);
        } else if (MODE == EPI_STATS_STORE16) {
          epilogue_stats_any<2>(p, &tma_c, es, tcol, mb, nb, quarter, lane);
        } else if (MODE == EPI_BF16) {
          epilogue_bf16(p, tcol, mb, nb, row);
        } else if (MODE == EPI_ACC_F32) {
          epilogue_out_f32<true>(p, &tma_c, es, tcol, mb, nb, quarter, lane);
        } else if (MODE == EPI_F32) {
          epilogue_out_f32<false>(p, &tma_c, es, tcol, mb, nb, quarter, lane);
        } else {
          epilogue_dz(p, tcol, mb, nb, row, coef);
        }
      }
      tc_fence_before_sync();
      mbar_arrive(&tempty[acc]);
      if (NBUF == 2) {
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      } else {
        acc_phase ^= 1u;
      }
    }
    // Outstanding bulk stores / reduce-adds must finish before the CTA exits.
    if ((MODE == EPI_STATS_STORE || MODE == EPI_STATS_STORE16 || MODE == EPI_ACC_F32 || MODE == EPI_F32) &&
        lane == 0)
      bulk_wait_group<0>();
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, 512);
  }
}

// ---------------------------------------------------------------------------
// CTA-pair variant: 256 x 256 tiles over a cluster of two CTAs on two SMs.
// Each CTA holds 128 rows of A and 128 of the 256 rows of B per K step (32 KB,
// a 6-stage ring), and one lane of the leader (cluster rank 0) issues
// tcgen05.mma.cta_group::2 with M = 256, N = 256, which reads both CTAs'
// shared memory and accumulates each CTA's 128 rows in its own TMEM. Each
// SM thus pulls the same operand bytes per flop as a single-CTA 256 x 256
// tile, while its accumulator is only 256 columns: two of them fit in TMEM,
// and the epilogue of one tile overlaps the MMAs of the next.
// Protocol: both CTAs wait on their own `empty` slot (the leader's MMA commit
// is multicast to both), load into their own ring, and count the bytes on the
// leader's `full` barrier, which the leader arms for both CTAs' bytes. The
// leader's accumulator commits are multicast to both CTAs' `tfull`; both
// CTAs' epilogue threads arrive on the leader's `tempty`. A cluster barrier
// after set-up and before teardown keeps either CTA from signalling a peer
// that is not there. Every mbarrier wait is bounded as in the kernel above.
constexpr int kPairStages = 6;

template <int MODE, bool A_MN, bool B_MN>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kGemmThreads, 1)
    gemm_tc_pair_kernel(const __grid_constant__ CUtensorMap tma_a, const __grid_constant__ CUtensorMap tma_b,
                        const __grid_constant__ CUtensorMap tma_c, const GemmParams p) {
  constexpr int S = kPairStages;
  constexpr int ABytes = kAStageBytes;      // 128 rows x 64 K
  constexpr int BBytes = kBStageBytes / 2;  // 128 of the tile's 256 B rows x 64 K
  static_assert(S * (ABytes + BBytes) <= kStages * (kAStageBytes + kBStageBytes), "ring exceeds the budget");
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  uint8_t* sA = smem;
  uint8_t* sB = smem + S * ABytes;
  uint8_t* sStage = smem + kStages * (kAStageBytes + kBStageBytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(sStage + kEpiStagingBytes);
  uint64_t* empty = full + S;
  uint64_t* tfull = empty + S;
  uint64_t* tempty = tfull + 2;
  uint64_t* mma_done = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 2 * 4);  // one arrival per epilogue warp of both CTAs (on the leader's)
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tma_a);
    tma_prefetch_desc(&tma_b);
    if (MODE == EPI_STATS_STORE || MODE == EPI_STATS_STORE16 || MODE == EPI_ACC_F32 || MODE == EPI_F32)
      tma_prefetch_desc(&tma_c);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, 512);  // one warp of each CTA, together
    tmem_relinquish_pair();
  }
  tc_fence_before_sync();
  cluster_sync_all();  // barriers initialised and TMEM allocated in both CTAs
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;

  const WaitCtx wc{abort_flag, p.status, p.timeout_ns};
  const int units_m = (p.m_tiles + 1) / 2;
  const int group = p.group_m / 2 > 0 ? p.group_m / 2 : 1;
  const int total = units_m * p.n_tiles;
  const int cluster = blockIdx.x >> 1;
  const int n_clusters = gridDim.x >> 1;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      const uint32_t full0 = mapa_shared(smem_u32(&full[0]), 0);  // the leader's full[0]
      int stage = 0;
      uint32_t phase = 0;
      bool aborted = false;
      if (!(p.debug_flags & FLCE_FLAG_TEST_STALL)) {
        for (int t = cluster; t < total && !aborted; t += n_clusters) {
          int mu, nb;
          tile_coords(p, units_m, group, t, mu, nb);
          const int row_a = p.a_row0 + (mu * 2 + static_cast<int>(rank)) * kBM;
          const int row_b = p.b_row0 + nb * kBN + static_cast<int>(rank) * (kBN / 2);
          for (int k = 0; k < p.k_iters; ++k) {
            if (!wait_bounded(&empty[stage], phase ^ 1u, wc)) {
              aborted = true;
              break;
            }
            if (rank == 0) mbar_arrive_expect_tx(&full[stage], 2 * (ABytes + BBytes));
            const uint32_t bar = full0 + static_cast<uint32_t>(stage) * 8u;
            if (A_MN) {
#pragma unroll
              for (int j = 0; j < kBM / 64; ++j)
                tma_load_2d_pair(sA + stage * ABytes + j * 8192, &tma_a, bar, row_a + j * 64, k * kBK);
            } else {
              tma_load_2d_pair(sA + stage * ABytes, &tma_a, bar, k * kBK, row_a);
            }
            if (B_MN) {
#pragma unroll
              for (int j = 0; j < (kBN / 2) / 64; ++j)
                tma_load_2d_pair(sB + stage * BBytes + j * 8192, &tma_b, bar, row_b + j * 64, k * kBK);
            } else {
              tma_load_2d_pair(sB + stage * BBytes, &tma_b, bar, k * kBK, row_b);
            }
            if (++stage == S) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (leader)
    if (lane == 0 && rank == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool aborted = false;
      constexpr uint32_t idesc = idesc_bf16_f32(2 * kBM, kBN, A_MN, B_MN);
      const uint32_t a_base = smem_u32(sA);
      const uint32_t b_base = smem_u32(sB);
      for (int t = cluster; t < total && !aborted; t += n_clusters) {
        if (!wait_bounded(&tempty[acc], acc_phase ^ 1u, wc)) break;
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kBN);
        for (int k = 0; k < p.k_iters; ++k) {
          if (!wait_bounded(&full[stage], phase, wc)) {
            aborted = true;
            break;
          }
          tc_fence_after_sync();
          const uint32_t a0 = a_base + stage * ABytes;
          const uint32_t b0 = b_base + stage * BBytes;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ad = A_MN ? sdesc_mnmajor_sw128(a0 + kk * 2048) : sdesc_kmajor_sw128(a0 + kk * 32);
            const uint64_t bd = B_MN ? sdesc_mnmajor_sw128(b0 + kk * 2048) : sdesc_kmajor_sw128(b0 + kk * 32);
            tc_mma_bf16_pair(d_tmem, ad, bd, idesc, (k | kk) != 0 ? 1u : 0u);
          }
          tc_commit_pair(&empty[stage], 0x3);
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (aborted) break;
        tc_commit_pair(&tfull[acc], 0x3);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      // All issued tensor-core work must finish before either CTA frees TMEM.
      tc_commit_pair(mma_done, 0x1);
      wait_drain(mma_done, 0, p.timeout_ns, p.status);
    }
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    float coef = 0.f;
    if (MODE == EPI_DZ) {
      const int64_t nv = p.hdr->n_valid;
      if (nv > 0) coef = p.reduction == FLCE_REDUCTION_MEAN ? p.grad_scale / static_cast<float>(nv) : p.grad_scale;
    }
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
    EpiStage es{sStage + (warp - 2) * 2 * kStageBufBytes, 0, 2, 0, p.store_hint != 0};
    if (es.hint) es.policy = l2_policy_evict_first();
    const uint32_t tempty0 = mapa_shared(smem_u32(&tempty[0]), 0);  // the leader's tempty[0]
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = cluster; t < total; t += n_clusters) {
      int mu, nb;
      tile_coords(p, units_m, group, t, mu, nb);
      bool ok = wait_bounded(&tfull[acc], acc_phase, wc);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after_sync();
      const int mb = mu * 2 + static_cast<int>(rank);
      if (mb < p.m_tiles) {
        const uint32_t tcol = t_lane + static_cast<uint32_t>(acc * kBN);
        if (MODE == EPI_STATS) {
          epilogue_stats_any<0>(p, &tma_c, es, tcol, mb, nb, quarter, lane);
        } else if (MODE == EPI_STATS_STORE) {
          epilogue_stats_any<1>(p, &tma_c, es, tcol, mb, nb, quarter, lane);
        } else if (MODE == EPI_STATS_STORE16) {
          epilogue_stats_any<2>(p, &tma_c, es, tcol, mb, nb, quarter, lane);
        } else if (MODE == EPI_BF16) {
          epilogue_bf16(p, tcol, mb, nb, row);
        } else if (MODE == EPI_ACC_F32) {
          epilogue_out_f32<true>(p, &tma_c, es, tcol, mb, nb, quarter, lane);
        } else if (MODE == EPI_F32) {
          epilogue_out_f32<false>(p, &tma_c, es, tcol, mb, nb, quarter, lane);
        } else {
          epilogue_dz(p, tcol, mb, nb, row, coef);
        }
      }
      // The warp's TMEM reads are complete (each thread waited for its loads);
      // one lane then arrives for the warp, which keeps the cross-SM arrivals
      // on the leader's barrier to four per CTA and tile.
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        if (rank == 0)
          mbar_arrive(&tempty[acc]);
        else
          mbar_arrive_cluster(tempty0 + static_cast<uint32_t>(acc) * 8u);
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if ((MODE == EPI_STATS_STORE || MODE == EPI_STATS_STORE16 || MODE == EPI_ACC_F32 || MODE == EPI_F32) &&
        lane == 0)
      bulk_wait_group<0>();
  }

  tc_fence_before_sync();
  cluster_sync_all();  // neither CTA leaves while the other may still signal it
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem_base, 512);
  }
}

template <int MODE, bool A_MN, bool B_MN>
static cudaError_t launch_mode_pair(const CUtensorMap* a, const CUtensorMap* b, const CUtensorMap* c,
                                    const GemmParams& p, int grid, cudaStream_t s) {
  static std::atomic<bool> configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(gemm_tc_pair_kernel<MODE, A_MN, B_MN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kGemmSmemBytes);
    if (e != cudaSuccess) return e;
    configured[dev].store(true, std::memory_order_release);
  }
  // one cluster of two CTAs per 256 x 256 tile at most, and an even grid
  const int units = ((p.m_tiles + 1) / 2) * p.n_tiles;
  int clusters = grid / 2;
  if (clusters > units) clusters = units;
  if (clusters < 1) clusters = 1;
  gemm_tc_pair_kernel<MODE, A_MN, B_MN><<<2 * clusters, kGemmThreads, kGemmSmemBytes, s>>>(*a, *b, c ? *c : *a, p);
  return cudaGetLastError();
}

template <int MODE, bool A_MN, bool B_MN, bool TF32 = false, int TMH = 1, bool SPLIT = false>
static cudaError_t launch_mode(const CUtensorMap* a, const CUtensorMap* b, const CUtensorMap* c,
                               const GemmParams& p, int grid, cudaStream_t s, const CUtensorMap* a2 = nullptr,
                               const CUtensorMap* b2 = nullptr) {
  // The shared-memory opt-in is a per-device function attribute: set it on the
  // first launch on each device (outside any stream capture that follows).
  // Two host threads may both set it on a first call; that is harmless, and
  // the flags are atomic so the check itself is not a data race.
  static std::atomic<bool> configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(gemm_tc_kernel<MODE, A_MN, B_MN, TF32, TMH, SPLIT>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmemBytes);
    if (e != cudaSuccess) return e;
    configured[dev].store(true, std::memory_order_release);
  }
  const int units = ((p.m_tiles + TMH - 1) / TMH) * p.n_tiles;
  if (grid > units) grid = units;
  if (grid < 1) grid = 1;
  gemm_tc_kernel<MODE, A_MN, B_MN, TF32, TMH, SPLIT><<<grid, gemm_threads(TMH), kGemmSmemBytes, s>>>(
      *a, *b, c ? *c : *a, a2 ? *a2 : *a, b2 ? *b2 : *b, p);
  return cudaGetLastError();
}

cudaError_t launch_gemm_tc(int mode, bool a_mn, bool b_mn, bool wide, const CUtensorMap* a, const CUtensorMap* b,
                           const CUtensorMap* c, const GemmParams& p, int grid, cudaStream_t s, bool pair) {
  if ((mode == EPI_STATS_STORE || mode == EPI_STATS_STORE16 || mode == EPI_ACC_F32 || mode == EPI_F32) &&
      c == nullptr)
    return cudaErrorInvalidValue;
  // pair: 256 x 256 tiles over CTA pairs (cta_group::2); a K-major B map must
  // then have 128-row boxes (each CTA loads half of the tile's B rows).
  if (wide && pair) {
    if (!a_mn && !b_mn) {
      switch (mode) {
        case EPI_STATS: return launch_mode_pair<EPI_STATS, false, false>(a, b, c, p, grid, s);
        case EPI_STATS_STORE: return launch_mode_pair<EPI_STATS_STORE, false, false>(a, b, c, p, grid, s);
        case EPI_STATS_STORE16: return launch_mode_pair<EPI_STATS_STORE16, false, false>(a, b, c, p, grid, s);
        case EPI_DZ: return launch_mode_pair<EPI_DZ, false, false>(a, b, c, p, grid, s);
        default: break;
      }
    }
    if (!a_mn && b_mn && mode == EPI_BF16) return launch_mode_pair<EPI_BF16, false, true>(a, b, c, p, grid, s);
    if (!a_mn && b_mn && mode == EPI_ACC_F32) return launch_mode_pair<EPI_ACC_F32, false, true>(a, b, c, p, grid, s);
    if (a_mn && b_mn && mode == EPI_ACC_F32) return launch_mode_pair<EPI_ACC_F32, true, true>(a, b, c, p, grid, s);
    return cudaErrorInvalidValue;
  }
  // The combinations the engine uses: the forward GEMM (both K-major), grad_h
  // (dz K-major, W MN-major or its transpose K-major), grad_W (dz and h_c
  // MN-major, or their transposes K-major).
  // wide: 256-row CTA tiles (TMH = 2) for every combination above except the
  // all-K-major backward cross-checks, which keep 128-row tiles.
  if (wide) {
    if (!a_mn && !b_mn) {
      switch (mode) {
        case EPI_STATS: return launch_mode<EPI_STATS, false, false, false, 2>(a, b, c, p, grid, s);
        case EPI_STATS_STORE: return launch_mode<EPI_STATS_STORE, false, false, false, 2>(a, b, c, p, grid, s);
        case EPI_STATS_STORE16:
          return launch_mode<EPI_STATS_STORE16, false, false, false, 2>(a, b, c, p, grid, s);
        case EPI_DZ: return launch_mode<EPI_DZ, false, false, false, 2>(a, b, c, p, grid, s);
        default: break;
      }
    }
    if (!a_mn && b_mn && mode == EPI_BF16) return launch_mode<EPI_BF16, false, true, false, 2>(a, b, c, p, grid, s);
    if (!a_mn && b_mn && mode == EPI_ACC_F32)
      return launch_mode<EPI_ACC_F32, false, true, false, 2>(a, b, c, p, grid, s);
    if (a_mn && b_mn && mode == EPI_ACC_F32) return launch_mode<EPI_ACC_F32, true, true, false, 2>(a, b, c, p, grid, s);
  }
  if (!a_mn && !b_mn) {
    switch (mode) {
      case EPI_STATS: return launch_mode<EPI_STATS, false, false>(a, b, c, p, grid, s);
      case EPI_STATS_STORE: return launch_mode<EPI_STATS_STORE, false, false>(a, b, c, p, grid, s);
      case EPI_STATS_STORE16: return launch_mode<EPI_STATS_STORE16, false, false>(a, b, c, p, grid, s);
      case EPI_BF16: return launch_mode<EPI_BF16, false, false>(a, b, c, p, grid, s);
      case EPI_ACC_F32: return launch_mode<EPI_ACC_F32, false, false>(a, b, c, p, grid, s);
      case EPI_DZ: return launch_mode<EPI_DZ, false, false>(a, b, c, p, grid, s);
      default: return cudaErrorInvalidValue;
    }
  }
  if (!a_mn && b_mn && mode == EPI_BF16) return launch_mode<EPI_BF16, false, true>(a, b, c, p, grid, s);
  if (!a_mn && b_mn && mode == EPI_ACC_F32) return launch_mode<EPI_ACC_F32, false, true>(a, b, c, p, grid, s);
  if (a_mn && b_mn && mode == EPI_ACC_F32) return launch_mode<EPI_ACC_F32, true, true>(a, b, c, p, grid, s);
  return cudaErrorInvalidValue;
}

cudaError_t launch_gemm_tc_tf32(int mode, bool wide, const CUtensorMap* a, const CUtensorMap* b,
                                const CUtensorMap* c, const GemmParams& p, int grid, cudaStream_t s,
                                const CUtensorMap* a_lo, const CUtensorMap* b_lo) {
  if ((mode == EPI_STATS_STORE || mode == EPI_ACC_F32 || mode == EPI_F32) && c == nullptr)
    return cudaErrorInvalidValue;
  if (a_lo != nullptr || b_lo != nullptr) {  // three-pass tf32, 128-row tiles
    if (a_lo == nullptr || b_lo == nullptr) return cudaErrorInvalidValue;
    switch (mode) {
      case EPI_STATS: return launch_mode<EPI_STATS, false, false, true, 1, true>(a, b, c, p, grid, s, a_lo, b_lo);
      case EPI_STATS_STORE:
        return launch_mode<EPI_STATS_STORE, false, false, true, 1, true>(a, b, c, p, grid, s, a_lo, b_lo);
      case EPI_F32: return launch_mode<EPI_F32, false, false, true, 1, true>(a, b, c, p, grid, s, a_lo, b_lo);
      case EPI_ACC_F32:
        return launch_mode<EPI_ACC_F32, false, false, true, 1, true>(a, b, c, p, grid, s, a_lo, b_lo);
      default: return cudaErrorInvalidValue;
    }
  }
  if (wide) {
    switch (mode) {
      case EPI_STATS: return launch_mode<EPI_STATS, false, false, true, 2>(a, b, c, p, grid, s);
      case EPI_STATS_STORE: return launch_mode<EPI_STATS_STORE, false, false, true, 2>(a, b, c, p, grid, s);
      case EPI_F32: return launch_mode<EPI_F32, false, false, true, 2>(a, b, c, p, grid, s);
      case EPI_ACC_F32: return launch_mode<EPI_ACC_F32, false, false, true, 2>(a, b, c, p, grid, s);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (mode) {
    case EPI_STATS: return launch_mode<EPI_STATS, false, false, true>(a, b, c, p, grid, s);
    case EPI_STATS_STORE: return launch_mode<EPI_STATS_STORE, false, false, true>(a, b, c, p, grid, s);
    case EPI_F32: return launch_mode<EPI_F32, false, false, true>(a, b, c, p, grid, s);
    case EPI_ACC_F32: return launch_mode<EPI_ACC_F32, false, false, true>(a, b, c, p, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace flce
