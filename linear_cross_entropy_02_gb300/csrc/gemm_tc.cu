// Persistent tcgen05 GEMM with fused epilogues: D [M, N] = A [M, K] * B [N, K]^T.
//
// One CTA per SM, 192 threads, warp-specialised:
//   warp 0      one lane issues TMA loads of 128x64 A and 256x64 B slices into a
//               4-stage shared-memory ring (128-byte swizzle);
//   warp 1      owns the 512 TMEM columns; one lane issues tcgen05.mma
//               (M=128, N=256, K=16 per instruction, fp32 accumulate) into one
//               of two 256-column accumulators, so the epilogue of tile t
//               overlaps the main loop of tile t+1;
//   warps 2-5   the epilogue: thread r of the 128 owns row r of the tile
//               (TMEM lane r), reads 32 columns at a time with tcgen05.ld and
//               applies the mode's epilogue.
// Epilogue modes: forward statistics of the linear cross-entropy (softcap,
// running max / sum of exponentials, argmax, label logit) with or without
// storing the capped logits; bf16 store of alpha*acc (grad_h); fp32
// accumulate-in-place of alpha*acc (grad_W += ...).
// Every wait is bounded (FLCE_ERR_TIMEOUT); on the way out the CTA drains the
// copies and MMAs it issued and frees TMEM.
#include <cuda_bf16.h>
#include <math.h>

#include "flce_device.cuh"
#include "flce_epilogue.cuh"

namespace flce {

// Grouped rasterisation: tiles walk group_m row-tiles at a time, row-tile
// fastest, so the CTAs resident at once share a few B slices and a few A
// slices in L2.
__device__ __forceinline__ void tile_coords(const GemmParams& p, int t, int& mb, int& nb) {
  const int per_group = p.group_m * p.n_tiles;
  const int g = t / per_group;
  const int first_m = g * p.group_m;
  const int gsize = min(p.m_tiles - first_m, p.group_m);
  const int local = t - g * per_group;
  mb = first_m + local % gsize;
  nb = local / gsize;
}

template <bool STORE>
__device__ __forceinline__ void epilogue_stats(const GemmParams& p, uint32_t tcol, int mb, int nb,
                                               int row) {
  const int grow = mb * kBM + row;
  const bool row_ok = grow < p.M_valid;
  const int64_t label = row_ok ? __ldg(p.labels + grow) : p.ignore_index;
  const int n0 = nb * kBN;
  const bool has_label = label != p.ignore_index && label >= n0 && label < n0 + kBN;
  RowStats st;
  row_stats_init(st, n0);
  float* zrow = STORE ? p.zbuf + static_cast<int64_t>(grow) * p.ldz + n0 : nullptr;
#pragma unroll 1
  for (int c = 0; c < kBN / 32; ++c) {
    uint32_t r[32];
    tmem_load_32cols(tcol + c * 32, r);
    tmem_load_wait();
    float s[32];
    const int col0 = n0 + c * 32;
#pragma unroll
    for (int j = 0; j < 32; ++j)
      s[j] = cap_logit(__uint_as_float(r[j]) * p.alpha, p.softcap, p.inv_softcap, col0 + j < p.N_valid);
    if (STORE && row_ok) {
      float4* dst = reinterpret_cast<float4*>(zrow + c * 32);
#pragma unroll
      for (int q = 0; q < 8; ++q) dst[q] = make_float4(s[4 * q], s[4 * q + 1], s[4 * q + 2], s[4 * q + 3]);
    }
    row_stats_update32(st, s, col0, has_label ? label : -1);
  }
  if (row_ok) {
    const int64_t o = static_cast<int64_t>(nb) * p.ldp + grow;
    p.part_max[o] = st.mx;
    p.part_sum[o] = st.sum;
    p.part_idx[o] = st.arg;
    if (has_label) p.tgt[grow] = st.tgt;
  }
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
#pragma unroll 1
  for (int c = 0; c < kBN / 32; ++c) {
    uint32_t r[32];
    tmem_load_32cols(tcol + c * 32, r);
    tmem_load_wait();
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
  }
}

__device__ __forceinline__ void epilogue_acc_f32(const GemmParams& p, uint32_t tcol, int mb, int nb,
                                                 int row) {
  const int grow = mb * kBM + row;
  const bool row_ok = grow < p.M_valid;
  const int n0 = nb * kBN;
  float* orow = static_cast<float*>(p.out) + static_cast<int64_t>(grow) * p.ldo + n0;
#pragma unroll 1
  for (int c = 0; c < kBN / 32; ++c) {
    uint32_t r[32];
    tmem_load_32cols(tcol + c * 32, r);
    tmem_load_wait();
#pragma unroll
    for (int g = 0; g < 8; ++g) {
      const int col = n0 + c * 32 + g * 4;
      if (row_ok && col < p.N_valid) {
        float4* dst = reinterpret_cast<float4*>(orow + c * 32 + g * 4);
        float4 o = *dst;
        o.x += __uint_as_float(r[g * 4 + 0]) * p.alpha;
        o.y += __uint_as_float(r[g * 4 + 1]) * p.alpha;
        o.z += __uint_as_float(r[g * 4 + 2]) * p.alpha;
        o.w += __uint_as_float(r[g * 4 + 3]) * p.alpha;
        *dst = o;
      }
    }
  }
}

template <int MODE>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tma_a, const __grid_constant__ CUtensorMap tma_b,
                   const GemmParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * kAStageBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + kStages * kBStageBytes);
  uint64_t* empty = full + kStages;
  uint64_t* tfull = empty + kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* mma_done = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 128);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tma_a);
    tma_prefetch_desc(&tma_b);
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
  const int total = p.m_tiles * p.n_tiles;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      bool aborted = false;
      if (!(p.debug_flags & FLCE_FLAG_TEST_STALL)) {
        for (int t = blockIdx.x; t < total && !aborted; t += gridDim.x) {
          int mb, nb;
          tile_coords(p, t, mb, nb);
          for (int k = 0; k < p.k_iters; ++k) {
            if (!wait_bounded(&empty[stage], phase ^ 1u, wc)) {
              aborted = true;
              break;
            }
            mbar_arrive_expect_tx(&full[stage], kAStageBytes + kBStageBytes);
            tma_load_2d(sA + stage * kAStageBytes, &tma_a, &full[stage], k * kBK, p.a_row0 + mb * kBM);
            tma_load_2d(sB + stage * kBStageBytes, &tma_b, &full[stage], k * kBK, p.b_row0 + nb * kBN);
            ++issued;
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      if (aborted) {
        // The most recent min(issued, kStages) loads may still be in flight:
        // wait for each to land before this CTA's shared memory goes away.
        const int n = issued < kStages ? issued : kStages;
        int s = stage;
        uint32_t ph = phase;
        for (int i = 0; i < n; ++i) {
          if (s == 0) {
            s = kStages - 1;
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
      constexpr uint32_t idesc = idesc_bf16_f32(kBM, kBN);
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
          const uint32_t a0 = a_base + stage * kAStageBytes;
          const uint32_t b0 = b_base + stage * kBStageBytes;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            tc_mma_bf16(d_tmem, sdesc_kmajor_sw128(a0 + kk * 32), sdesc_kmajor_sw128(b0 + kk * 32), idesc,
                        (k | kk) != 0 ? 1u : 0u);
          }
          tc_commit(&empty[stage]);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (aborted) break;
        tc_commit(&tfull[acc]);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      // All issued tensor-core work must finish before TMEM is released.
      tc_commit(mma_done);
      wait_drain(mma_done, 0, p.timeout_ns, p.status);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;  // TMEM lanes this warp may access
    const int row = quarter * 32 + lane;
    const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      int mb, nb;
      tile_coords(p, t, mb, nb);
      bool ok = wait_bounded(&tfull[acc], acc_phase, wc);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after_sync();
      const uint32_t tcol = t_lane + static_cast<uint32_t>(acc * kBN);
      if (MODE == EPI_STATS) {
        epilogue_stats<false>(p, tcol, mb, nb, row);
      } else if (MODE == EPI_STATS_STORE) {
        epilogue_stats<true>(p, tcol, mb, nb, row);
      } else if (MODE == EPI_BF16) {
        epilogue_bf16(p, tcol, mb, nb, row);
      } else {
        epilogue_acc_f32(p, tcol, mb, nb, row);
      }
      tc_fence_before_sync();
      mbar_arrive(&tempty[acc]);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, 512);
  }
}

template <int MODE>
static cudaError_t launch_mode(const CUtensorMap* a, const CUtensorMap* b, const GemmParams& p, int grid,
                               cudaStream_t s) {
  // Per device and cheap: set on every launch rather than caching per process.
  cudaError_t e =
      cudaFuncSetAttribute(gemm_tc_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmemBytes);
  if (e != cudaSuccess) return e;
  gemm_tc_kernel<MODE><<<grid, kGemmThreads, kGemmSmemBytes, s>>>(*a, *b, p);
  return cudaGetLastError();
}

cudaError_t launch_gemm_tc(int mode, const CUtensorMap* a, const CUtensorMap* b, const GemmParams& p, int grid,
                           cudaStream_t s) {
  switch (mode) {
    case EPI_STATS: return launch_mode<EPI_STATS>(a, b, p, grid, s);
    case EPI_STATS_STORE: return launch_mode<EPI_STATS_STORE>(a, b, p, grid, s);
    case EPI_BF16: return launch_mode<EPI_BF16>(a, b, p, grid, s);
    case EPI_ACC_F32: return launch_mode<EPI_ACC_F32>(a, b, p, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace flce
