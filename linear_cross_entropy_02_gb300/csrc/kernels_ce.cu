// Cross-entropy on materialised logits [N, V] (bf16 or fp32): the non-fused
// branch next to the fused path (Liger-Kernel "Muse Glimmer" page, Testing Done:
// the non-fused softcap branch; DeepSeek-V3 page, Summary: logits kept outside
// training-with-labels). Both kernels stream the logits once each, coalesced:
//   ce_stats   one warp per (row, 8192-column tile), four 8-column loads in
//              flight per lane: max / sum of exponentials / first argmax per
//              lane, merged across the warp with shuffles; the lane holding the
//              label writes its capped logit.
//   ce_grad    one thread per 8 consecutive columns: recomputes s = cap(m x),
//              writes dL/dx = m c_i (exp(s - lse_i) - [j = y_i]) (1 - (s/T)^2).
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

// One warp per (row, 8192-column tile), eight warps per block, no block-level
// synchronisation. Per step the lane loads four 8-column pieces 256 columns
// apart (four loads in flight, each covering 512 B per warp), so a step spans
// 1024 columns and eight steps the tile; max / sum of exponentials / first
// argmax per lane, merged across the warp with shuffles.
template <typename T>
__global__ void __launch_bounds__(256) ce_stats_kernel(const CeParams p) {
  const int64_t task = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int row = static_cast<int>(task / p.n_vtiles);
  const int tile = static_cast<int>(task - static_cast<int64_t>(row) * p.n_vtiles);
  if (row >= p.rows) return;
  const T* x = static_cast<const T*>(p.logits) + static_cast<int64_t>(row) * p.ldx;
  const int64_t label = p.labels[row];
  const int c_begin = tile * kCeTile;
  const int c_end = min(c_begin + kCeTile, p.vocab);
  float m = -INFINITY, s = 0.f;
  int ix = c_begin;
  for (int base = c_begin; base < c_end; base += 1024) {
    float v[4][8];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int c0 = base + q * 256 + lane * 8;
      if (c0 + 8 <= c_end && p.vec_ok) {
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
      const int c0 = base + q * 256 + lane * 8;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const bool in = c0 + j < c_end;
        const float sv = in ? cap(v[q][j] * p.out_mult, p.softcap, p.inv_softcap) : -INFINITY;
        v[q][j] = sv;
        if (in && static_cast<int64_t>(c0 + j) == label) p.tgt[row] = sv;
        if (sv > cm) {  // columns go up with (q, j): the first maximum is kept
          cm = sv;
          ci = c0 + j;
        }
      }
    }
    if (cm > m) {
      s = (m == -INFINITY) ? 0.f : s * __expf(m - cm);
      m = cm;
      ix = ci;
    }
    if (m != -INFINITY) {
#pragma unroll
      for (int q = 0; q < 4; ++q)
#pragma unroll
        for (int j = 0; j < 8; ++j) s += __expf(v[q][j] - m);
    }
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

template <typename T>
__global__ void __launch_bounds__(256) ce_grad_kernel(const CeParams p) {
  const int row = blockIdx.y;
  const int c0 = (blockIdx.x * blockDim.x + threadIdx.x) * 8;
  if (row >= p.rows || c0 >= p.vocab) return;
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
  const float lse = p.lse[row];
  const float cm = c * p.out_mult;
  const T* x = static_cast<const T*>(p.logits) + static_cast<int64_t>(row) * p.ldx;
  T* g = static_cast<T*>(p.grad) + static_cast<int64_t>(row) * p.ldg;
  float v[8];
  const bool full = c0 + 8 <= p.vocab && p.vec_ok;
  if (full) {
    Vec8<T>::load(x + c0, v);
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = (c0 + j < p.vocab) ? Vec8<T>::load1(x + c0 + j) : 0.f;
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float sv = cap(v[j] * p.out_mult, p.softcap, p.inv_softcap);
    float q = __expf(sv - lse) - (static_cast<int64_t>(c0 + j) == label ? 1.f : 0.f);
    if (p.softcap > 0.f) {
      const float u = sv * p.inv_softcap;
      q *= (1.f - u * u);
    }
    v[j] = cm * q;
  }
  if (full) {
    Vec8<T>::store(g + c0, v);
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (c0 + j < p.vocab) Vec8<T>::store1(g + c0 + j, v[j]);
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
  dim3 grid((p.vocab + 2047) / 2048, p.rows);
  if (p.dtype == FLCE_DTYPE_BF16)
    ce_grad_kernel<uint16_t><<<grid, 256, 0, s>>>(p);
  else
    ce_grad_kernel<float><<<grid, 256, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace flce
