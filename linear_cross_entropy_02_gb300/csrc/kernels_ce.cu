// Cross-entropy on materialised logits [N, V] (bf16 or fp32): the non-fused
// branch next to the fused path (Liger-Kernel "Muse Glimmer" page, Testing Done:
// the non-fused softcap branch; DeepSeek-V3 page, Summary: logits kept outside
// training-with-labels). Both kernels stream the logits once each, coalesced:
//   ce_stats   one warp per (row, 8192-column tile), four 8-column loads in
//              flight per lane: max / sum of exponentials / first argmax per
//              lane, merged across the warp with shuffles; the lane holding the
//              label writes its capped logit.
//   ce_grad    one block per 8192 columns of a row, four 8-column pieces per
//              thread: recomputes s = cap(m x), writes
//              dL/dx = m c_i (exp(s - lse_i) - [j = y_i]) (1 - (s/T)^2).
// The per-tile statistics go through the same merge kernel as the fused path.
#include <cuda_bf16.h>
#include <math.h>

#include "flce_internal.h"

namespace flce {

namespace {

template <typename T>
struct Vec8;

template <>
struct Vec8<uint16_t> {  // bf16 bits
  static __device__ __forceinline__ void load(const uint16_t* p, float (&v)[8]) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = __uint_as_float(w[i] << 16);
      v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
  static __device__ __forceinline__ float load1(const uint16_t* p) {
    return __uint_as_float(static_cast<uint32_t>(*p) << 16);
  }
  static __device__ __forceinline__ void store(uint16_t* p, const float (&v)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat162 b = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
      w[i] = *reinterpret_cast<const uint32_t*>(&b);
    }
    *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
  }
  static __device__ __forceinline__ void store1(uint16_t* p, float v) {
    const __nv_bfloat16 b = __float2bfloat16_rn(v);
    *p = *reinterpret_cast<const uint16_t*>(&b);
  }
};

template <>
struct Vec8<float> {
  static __device__ __forceinline__ void load(const float* p, float (&v)[8]) {
    const float4 a = *reinterpret_cast<const float4*>(p);
    const float4 b = *reinterpret_cast<const float4*>(p + 4);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
  static __device__ __forceinline__ float load1(const float* p) { return *p; }
  static __device__ __forceinline__ void store(float* p, const float (&v)[8]) {
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
    *reinterpret_cast<float4*>(p + 4) = make_float4(v[4], v[5], v[6], v[7]);
  }
  static __device__ __forceinline__ void store1(float* p, float v) { *p = v; }
};

__device__ __forceinline__ float cap(float z, float softcap, float inv_softcap) {
  return softcap > 0.f ? softcap * tanhf(z * inv_softcap) : z;
}

// (max, sum of exp(x - max), index of first max) of two disjoint column sets.
__device__ __forceinline__ void merge_stats(float& m, float& s, int& ix, float m2, float s2, int ix2) {
  const float M = fmaxf(m, m2);
  if (M == -INFINITY) return;  // both empty
  s = s * __expf(m - M) + s2 * __expf(m2 - M);
  if (m2 > m || (m2 == m && ix2 < ix)) ix = ix2;
  m = M;
}

}  // namespace

constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float ex2f_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Per-lane statistics of one step: four 8-column pieces 256 columns apart.
// FULL: every column is inside the tile; CAP: softcap on. The label is found
// once per warp task, not per element (its lane writes it separately).
template <typename T, bool FULL, bool CAP>
__device__ __forceinline__ void ce_step(const CeParams& p, const T* x, int base, int c_end, int lane, float& m,
                                        float& s, int& ix) {
  float v[4][8];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int c0 = base + q * 256 + lane * 8;
    if (FULL && p.vec_ok) {
      Vec8<T>::load(x + c0, v[q]);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) v[q][j] = (c0 + j < c_end) ? Vec8<T>::load1(x + c0 + j) : 0.f;
    }
  }
  float cm = -INFINITY;
  int ci = 0;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      float sv = v[q][j] * p.out_mult;
      if (CAP) sv = p.softcap * tanhf(sv * p.inv_softcap);
      if (!FULL && base + q * 256 + lane * 8 + j >= c_end) sv = -INFINITY;
      v[q][j] = sv;
      if (sv > cm) {  // columns go up with (q, j): the first maximum is kept
        cm = sv;
        ci = q * 256 + j;
      }
    }
  }
  if (cm > m) {
    s = (m == -INFINITY) ? 0.f : s * ex2f_approx((m - cm) * kLog2e);
    m = cm;
    ix = base + lane * 8 + ci;
  }
  if (m != -INFINITY) {
    const float ml = m * kLog2e;
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
      for (int j = 0; j < 8; ++j) s += ex2f_approx(fmaf(v[q][j], kLog2e, -ml));
  }
}

// One warp per (row, 8192-column tile), eight warps per block, no block-level
// synchronisation: eight steps of 1024 columns, each with four 16- or 32-byte
// loads per lane in flight, max / sum of exponentials / first argmax per lane,
// then a shuffle merge across the warp.
template <typename T>
__global__ void __launch_bounds__(256) ce_stats_kernel(const CeParams p) {
  const int task = static_cast<int>((static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  const int row = task / p.n_vtiles;
  const int tile = task - row * p.n_vtiles;
  if (row >= p.rows) return;
  const T* x = static_cast<const T*>(p.logits) + static_cast<int64_t>(row) * p.ldx;
  const int c_begin = tile * kCeTile;
  const int c_end = min(c_begin + kCeTile, p.vocab);
  float m = -INFINITY, s = 0.f;
  int ix = c_begin;
  for (int base = c_begin; base < c_end; base += 1024) {
    const bool full = base + 1024 <= c_end;
    if (p.softcap > 0.f) {
      if (full)
        ce_step<T, true, true>(p, x, base, c_end, lane, m, s, ix);
      else
        ce_step<T, false, true>(p, x, base, c_end, lane, m, s, ix);
    } else {
      if (full)
        ce_step<T, true, false>(p, x, base, c_end, lane, m, s, ix);
      else
        ce_step<T, false, false>(p, x, base, c_end, lane, m, s, ix);
    }
  }
  // The label's capped logit, written by the lane that read that column (the
  // same arithmetic on a re-read of the one element).
  const int64_t label = p.labels[row];
  if (label >= c_begin && label < c_end) {
    const int d = static_cast<int>(label - c_begin);
    if (((d >> 3) & 31) == lane) p.tgt[row] = cap(Vec8<T>::load1(x + label) * p.out_mult, p.softcap, p.inv_softcap);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
    const int ix2 = __shfl_xor_sync(0xffffffffu, ix, o);
    merge_stats(m, s, ix, m2, s2, ix2);
  }
  if (lane == 0) {
    const int64_t o = static_cast<int64_t>(tile) * p.ldp + row;
    p.part_max[o] = m;
    p.part_sum[o] = s;
    p.part_idx[o] = ix;
  }
}

template <typename T, bool CAP>
__device__ __forceinline__ void ce_grad8(const CeParams& p, const T* x, T* g, int c0, bool full, float lse_l2e,
                                         float cm, int label_local) {
  float v[8];
  if (full) {
    Vec8<T>::load(x + c0, v);
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = (c0 + j < p.vocab) ? Vec8<T>::load1(x + c0 + j) : 0.f;
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    float sv = v[j] * p.out_mult;
    float cap_d = 1.f;
    if (CAP) {
      sv = p.softcap * tanhf(sv * p.inv_softcap);
      const float u = sv * p.inv_softcap;
      cap_d = 1.f - u * u;
    }
    const float q = ex2f_approx(fmaf(sv, kLog2e, -lse_l2e)) - (j == label_local ? 1.f : 0.f);
    v[j] = CAP ? cm * q * cap_d : cm * q;
  }
  if (full) {
    Vec8<T>::store(g + c0, v);
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (c0 + j < p.vocab) Vec8<T>::store1(g + c0 + j, v[j]);
  }
}

// A block covers 8192 columns of one row; thread t handles four 8-column
// pieces 2048 i + 8 t: recomputes s = cap(m x) and writes
// dL/dx = m c_i (exp(s - lse_i) - [j = y_i]) (1 - (s/T)^2).
template <typename T>
__global__ void __launch_bounds__(256) ce_grad_kernel(const CeParams p) {
  const int row = blockIdx.y;
  const int c_base = blockIdx.x * 8192 + threadIdx.x * 8;
  if (row >= p.rows || c_base >= p.vocab) return;
  const int64_t label = p.labels[row];
  const bool valid = label != p.ignore_index;
  const int64_t n_valid = p.hdr->n_valid;
  float c;
  if (!valid) {
    c = 0.f;
  } else if (p.reduction == FLCE_REDUCTION_NONE) {
    c = p.row_scale ? p.row_scale[row] : 1.f;
  } else if (n_valid == 0) {
    c = 0.f;
  } else {
    c = p.reduction == FLCE_REDUCTION_MEAN ? p.grad_scale / static_cast<float>(n_valid) : p.grad_scale;
  }
  const float lse_l2e = p.lse[row] * kLog2e;
  const float cm = c * p.out_mult;
  const T* x = static_cast<const T*>(p.logits) + static_cast<int64_t>(row) * p.ldx;
  T* g = static_cast<T*>(p.grad) + static_cast<int64_t>(row) * p.ldg;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int c0 = c_base + i * 2048;
    if (c0 >= p.vocab) break;
    const int64_t dl = valid ? label - c0 : -1;
    const int label_local = (dl >= 0 && dl < 8) ? static_cast<int>(dl) : -1;
    const bool full = c0 + 8 <= p.vocab && p.vec_ok;
    if (p.softcap > 0.f)
      ce_grad8<T, true>(p, x, g, c0, full, lse_l2e, cm, label_local);
    else
      ce_grad8<T, false>(p, x, g, c0, full, lse_l2e, cm, label_local);
  }
}

cudaError_t launch_ce_stats(const CeParams& p, cudaStream_t s) {
  if (p.rows <= 0) return cudaSuccess;
  const int64_t warps = static_cast<int64_t>(p.rows) * p.n_vtiles;
  const unsigned blocks = static_cast<unsigned>((warps + 7) / 8);
  if (p.dtype == FLCE_DTYPE_BF16)
    ce_stats_kernel<uint16_t><<<blocks, 256, 0, s>>>(p);
  else
    ce_stats_kernel<float><<<blocks, 256, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_ce_grad(const CeParams& p, cudaStream_t s) {
  if (p.rows <= 0) return cudaSuccess;
  dim3 grid((p.vocab + 8191) / 8192, p.rows);
  if (p.dtype == FLCE_DTYPE_BF16)
    ce_grad_kernel<uint16_t><<<grid, 256, 0, s>>>(p);
  else
    ce_grad_kernel<float><<<grid, 256, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace flce
