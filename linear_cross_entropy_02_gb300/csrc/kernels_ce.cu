// Cross-entropy on materialised logits [N, V] (bf16 or fp32): the non-fused
// branch next to the fused path (Liger-Kernel "Muse Glimmer" page, Testing Done:
// the non-fused softcap branch; DeepSeek-V3 page, Summary: logits kept outside
// training-with-labels). Both kernels stream the logits once each, coalesced:
//   ce_stats   one block per (row, 2048-column tile), 8 columns per thread:
//              max / sum of exponentials / first argmax per thread, merged
//              with shuffles and across warps in a fixed order; the thread
//              holding the label writes its capped logit.
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

// One 256-thread block per (row, 2048-column tile): thread t holds columns
// 8t .. 8t+7 of the tile (one 16- or 32-byte load, coalesced across the block,
// the same pattern as the gradient kernel); per-thread max / sum / first argmax,
// merged across each warp with shuffles and across the 8 warps in warp order.
template <typename T>
__global__ void __launch_bounds__(256) ce_stats_kernel(const CeParams p) {
  __shared__ float s_m[8];
  __shared__ float s_s[8];
  __shared__ int s_i[8];
  const int row = blockIdx.y;
  const int tile = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const T* x = static_cast<const T*>(p.logits) + static_cast<int64_t>(row) * p.ldx;
  const int64_t label = p.labels[row];
  const int c_begin = tile * kCeTile;
  const int c_end = min(c_begin + kCeTile, p.vocab);
  const int c0 = c_begin + threadIdx.x * 8;
  float v[8];
  if (c0 + 8 <= c_end && p.vec_ok) {
    Vec8<T>::load(x + c0, v);
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = (c0 + j < c_end) ? Vec8<T>::load1(x + c0 + j) : 0.f;
  }
  float m = -INFINITY, s = 0.f;
  int ix = c0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const bool in = c0 + j < c_end;
    const float sv = in ? cap(v[j] * p.out_mult, p.softcap, p.inv_softcap) : -INFINITY;
    v[j] = sv;
    if (in && static_cast<int64_t>(c0 + j) == label) p.tgt[row] = sv;
    if (sv > m) {
      m = sv;
      ix = c0 + j;
    }
  }
  if (m != -INFINITY) {
#pragma unroll
    for (int j = 0; j < 8; ++j) s += __expf(v[j] - m);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
    const int ix2 = __shfl_xor_sync(0xffffffffu, ix, o);
    merge_stats(m, s, ix, m2, s2, ix2);
  }
  if (lane == 0) {
    s_m[warp] = m;
    s_s[warp] = s;
    s_i[warp] = ix;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float M = s_m[0], S = s_s[0];
    int I = s_i[0];
    for (int w = 1; w < 8; ++w) merge_stats(M, S, I, s_m[w], s_s[w], s_i[w]);
    const int64_t o = static_cast<int64_t>(tile) * p.ldp + row;
    p.part_max[o] = M;
    p.part_sum[o] = S;
    p.part_idx[o] = I;
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
  dim3 grid(p.n_vtiles, p.rows);
  if (p.dtype == FLCE_DTYPE_BF16)
    ce_stats_kernel<uint16_t><<<grid, 256, 0, s>>>(p);
  else
    ce_stats_kernel<float><<<grid, 256, 0, s>>>(p);
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
