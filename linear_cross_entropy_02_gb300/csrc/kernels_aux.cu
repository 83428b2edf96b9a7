// The bandwidth-bound and bookkeeping kernels of the fused linear cross-entropy
// path, plus the debug fp32-FMA GEMM:
//   prologue      label check, n_valid, reset of the device scalars
//   merge         per-row merge of the vocab-tile statistics: lse, argmax,
//                 row loss; fixed-order reduction into the batch sums; or one
//                 vocab shard's per-row partials
//   vp merge      the merge of every vocab shard's partials, in shard order
//   dlogits       dz = c (softmax - onehot) (1 - (s/T)^2) in bf16 from the
//                 stored logits (fp16 s - gmax, or fp32), row-major (A operand
//                 of grad_h, and MN-major A of grad_W), and on the K-major
//                 paths also transposed; fp32 (and its tf32 split) on the
//                 fp32-operand path
//   transpose     bf16 / fp32 transposes that give the backward GEMMs K-major
//                 operands; split: the hi / lo halves of the three-pass tf32
//   finish        loss and token accuracy scalars
//   scale         y = scale * x with a dtype conversion (autograd's backward)
//   simt gemm     fp32 FMA GEMM + statistics from stored logits (debug path)
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include "flce_device.cuh"
#include "flce_epilogue.cuh"
#include "flce_internal.h"

namespace flce {

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

__device__ __forceinline__ uint16_t float_to_bf16_bits(float f) {
  const __nv_bfloat16 v = __float2bfloat16_rn(f);
  return *reinterpret_cast<const uint16_t*>(&v);
}

// x = hi + lo with hi = x rounded to tf32 (10 mantissa bits, nearest, ties
// away from zero: cvt.rna.tf32.f32) and lo = x - hi, exact in fp32: the two
// operands of the three-pass tf32 products.
__device__ __forceinline__ void split_tf32(float x, float& hi, float& lo) {
  uint32_t h;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(h) : "f"(x));
  hi = __uint_as_float(h);
  lo = x - hi;
}

// ------------------------------------------------------------------ prologue
// One block: counts rows whose label is not ignore_index, flags labels outside
// [0, V), and resets the batch sums. Deterministic (no atomics).
__global__ void __launch_bounds__(1024) prologue_kernel(const int64_t* __restrict__ labels, int64_t n,
                                                        int64_t vocab, int64_t ignore_index, Header* hdr) {
  __shared__ long long s_cnt[32];
  __shared__ int s_bad[32];
  long long cnt = 0;
  int bad = 0;
  for (int64_t i = threadIdx.x; i < n; i += blockDim.x) {
    const int64_t y = labels[i];
    if (y != ignore_index) {
      ++cnt;
      if (y < 0 || y >= vocab) bad = 1;
    }
  }
  for (int o = 16; o > 0; o >>= 1) {
    cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
    bad |= __shfl_xor_sync(0xffffffffu, bad, o);
  }
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) {
    s_cnt[w] = cnt;
    s_bad[w] = bad;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    long long c = 0;
    int b = 0;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) {
      c += s_cnt[i];
      b |= s_bad[i];
    }
    hdr->status = b ? FLCE_ERR_LABEL : 0;
    hdr->ticket = 0;
    hdr->n_valid = c;
    hdr->loss_sum = 0.0;
    hdr->correct = 0;
  }
}

cudaError_t launch_prologue(const int64_t* labels, int64_t n, int64_t vocab, int64_t ignore_index, Header* hdr,
                            cudaStream_t s) {
  prologue_kernel<<<1, 1024, 0, s>>>(labels, n, vocab, ignore_index, hdr);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ merge
// 32 rows per block (one per lane) x 8 warps: warp w folds vocab tiles w, w+8,
// w+16, ... of its lane's row (reads of one tile are 32 consecutive rows), the
// eight partial results are merged in warp order through shared memory, and
// warp 0 finishes the rows. Ties keep the lowest vocab index throughout.
constexpr int kMergeWarps = 8;

__global__ void __launch_bounds__(kMergeRows * kMergeWarps) merge_kernel(const MergeParams p) {
  __shared__ float s_m[kMergeWarps][kMergeRows];
  __shared__ float s_s[kMergeWarps][kMergeRows];
  __shared__ int s_a[kMergeWarps][kMergeRows];
  __shared__ bool s_last;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int row = blockIdx.x * kMergeRows + lane;
  float mx = -INFINITY, sum = 0.f;
  int arg = 0x7fffffff;
  if (row < p.rows) {
    for (int t = warp; t < p.n_vtiles; t += kMergeWarps) {
      const int64_t o = static_cast<int64_t>(t) * p.ldp + row;
      const float pm = p.part_max[o];
      const float ps = p.part_sum[o];
      if (pm > mx) {
        sum = sum * expf(mx - pm) + ps;
        mx = pm;
        arg = p.part_idx[o];
      } else {
        sum += ps * expf(pm - mx);
      }
    }
  }
  s_m[warp][lane] = mx;
  s_s[warp][lane] = sum;
  s_a[warp][lane] = arg;
  __syncthreads();
  if (p.shard_out != nullptr) {
    // one vocab shard's partials; the batch sums wait for the merge of all shards
    if (warp == 0 && row < p.rows) {
      float M = -INFINITY, S = 0.f;
      int A = 0x7fffffff;
      for (int w = 0; w < kMergeWarps; ++w) {
        const float m2 = s_m[w][lane];
        const float s2 = s_s[w][lane];
        const int a2 = s_a[w][lane];
        if (m2 == -INFINITY) continue;
        if (m2 > M) {
          S = S * expf(M - m2) + s2;
          M = m2;
          A = a2;
        } else {
          S += s2 * expf(m2 - M);
          if (m2 == M && a2 < A) A = a2;
        }
      }
      if (!isfinite(M) || !isfinite(S)) atomicOr(&p.hdr->status, FLCE_ERR_NONFINITE);
      const int64_t y = p.labels[row];
      const int64_t yl = y - p.vocab_offset;
      const bool here = y != p.ignore_index && yl >= 0 && yl < p.vocab_shard;
      p.shard_out[row] = M;
      p.shard_out[p.ld_shard + row] = S;
      p.shard_out[2 * p.ld_shard + row] = __int_as_float(static_cast<int>(A + p.vocab_offset));
      p.shard_out[3 * p.ld_shard + row] = here ? p.tgt[row] : 0.f;
    }
    return;
  }
  if (warp == 0) {
    double loss_i = 0.0;
    long long corr_i = 0;
    if (row < p.rows) {
      float M = -INFINITY, S = 0.f;
      int A = 0x7fffffff;
      for (int w = 0; w < kMergeWarps; ++w) {
        const float m2 = s_m[w][lane];
        const float s2 = s_s[w][lane];
        const int a2 = s_a[w][lane];
        if (m2 == -INFINITY) continue;
        if (m2 > M) {
          S = S * expf(M - m2) + s2;
          M = m2;
          A = a2;
        } else {
          S += s2 * expf(m2 - M);
          if (m2 == M && a2 < A) A = a2;
        }
      }
      const float lse = M + logf(S);
      p.lse[row] = lse;
      if (!isfinite(lse)) {  // inf / NaN inputs: no meaningful argmax
        atomicOr(&p.hdr->status, FLCE_ERR_NONFINITE);
        A = -1;
      }
      const int64_t y = p.labels[row];
      if (y != p.ignore_index) {
        loss_i = static_cast<double>(lse) - static_cast<double>(p.tgt[row]);
        corr_i = (static_cast<int64_t>(A) == y) ? 1 : 0;
      }
      if (p.predicted) p.predicted[row] = A;
      if (p.row_lse) p.row_lse[row] = lse;
      if (p.row_loss) p.row_loss[row] = static_cast<float>(loss_i);
    }
    for (int o = 16; o > 0; o >>= 1) {
      loss_i += __shfl_xor_sync(0xffffffffu, loss_i, o);
      corr_i += __shfl_xor_sync(0xffffffffu, corr_i, o);
    }
    if (lane == 0) {
      p.block_loss[blockIdx.x] = loss_i;
      p.block_correct[blockIdx.x] = corr_i;
      __threadfence();
      const unsigned int ticket = atomicAdd(&p.hdr->ticket, 1u);
      s_last = (ticket == gridDim.x - 1);
    }
  }
  __syncthreads();
  // The last block to finish adds the block sums in block order, so the result
  // does not depend on which block finished when.
  if (s_last && threadIdx.x == 0) {
    __threadfence();
    double tl = 0.0;
    long long tc = 0;
    for (unsigned int b = 0; b < gridDim.x; ++b) {
      tl += reinterpret_cast<volatile double*>(p.block_loss)[b];
      tc += reinterpret_cast<volatile long long*>(p.block_correct)[b];
    }
    p.hdr->loss_sum += tl;
    p.hdr->correct += tc;
    p.hdr->ticket = 0;
  }
}

cudaError_t launch_merge(const MergeParams& p, cudaStream_t s) {
  const int blocks = (p.rows + kMergeRows - 1) / kMergeRows;
  if (blocks == 0) return cudaSuccess;
  merge_kernel<<<blocks, kMergeRows * kMergeWarps, 0, s>>>(p);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ vocab-shard merge
// One warp of 32 rows per block. Row i folds the partials of shards 0..S-1 in
// order: the running max is replaced only on a strict increase, so on ties the
// lower shard (the lower vocab ids) keeps the argmax, as within a shard. The
// label's logit comes from the shard whose range holds the label.
__global__ void __launch_bounds__(32) vp_merge_kernel(const VpMergeParams p) {
  const int lane = threadIdx.x;
  const int row = blockIdx.x * 32 + lane;
  double loss_i = 0.0;
  long long corr_i = 0;
  if (row < p.rows) {
    float M = -INFINITY, S = 0.f;
    int A = 0x7fffffff;
    for (int k = 0; k < p.n_shards; ++k) {
      const float* q = p.partials + static_cast<int64_t>(k) * 4 * p.ld;
      const float m2 = q[row];
      const float s2 = q[p.ld + row];
      const int a2 = __float_as_int(q[2 * p.ld + row]);
      if (m2 == -INFINITY) continue;
      if (m2 > M) {
        S = S * expf(M - m2) + s2;
        M = m2;
        A = a2;
      } else {
        S += s2 * expf(m2 - M);
      }
    }
    const float lse = M + logf(S);
    p.lse[row] = lse;
    if (!isfinite(lse)) {
      atomicOr(&p.hdr->status, FLCE_ERR_NONFINITE);
      A = -1;
    }
    const int64_t y = p.labels[row];
    if (y != p.ignore_index) {
      int k = 0;
      while (k + 1 < p.n_shards && y >= p.offsets[k + 1]) ++k;
      const float t = p.partials[static_cast<int64_t>(k) * 4 * p.ld + 3 * p.ld + row];
      loss_i = static_cast<double>(lse) - static_cast<double>(t);
      corr_i = (static_cast<int64_t>(A) == y) ? 1 : 0;
    }
    if (p.predicted) p.predicted[row] = A;
    if (p.row_lse) p.row_lse[row] = lse;
  }
  for (int o = 16; o > 0; o >>= 1) {
    loss_i += __shfl_xor_sync(0xffffffffu, loss_i, o);
    corr_i += __shfl_xor_sync(0xffffffffu, corr_i, o);
  }
  unsigned int last = 0;
  if (lane == 0) {
    p.block_loss[blockIdx.x] = loss_i;
    p.block_correct[blockIdx.x] = corr_i;
    __threadfence();
    last = atomicAdd(&p.hdr->ticket, 1u) == gridDim.x - 1;
  }
  // the last block adds the block sums in block order (a fixed order)
  if (lane == 0 && last) {
    __threadfence();
    double tl = 0.0;
    long long tc = 0;
    for (unsigned int b = 0; b < gridDim.x; ++b) {
      tl += reinterpret_cast<volatile double*>(p.block_loss)[b];
      tc += reinterpret_cast<volatile long long*>(p.block_correct)[b];
    }
    p.hdr->loss_sum += tl;
    p.hdr->correct += tc;
    p.hdr->ticket = 0;
  }
}

cudaError_t launch_vp_merge(const VpMergeParams& p, cudaStream_t s) {
  const int blocks = (p.rows + 31) / 32;
  if (blocks == 0) return cudaSuccess;
  vp_merge_kernel<<<blocks, 32, 0, s>>>(p);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ dlogits
// 64x64 tile per 256-thread block. Thread (ty, tx) handles rows ty + 16 k and
// columns 4 tx .. 4 tx + 3, so reads of s (fp32) and writes of dz (bf16) are
// contiguous along a row; the transposed copy goes through shared memory.
constexpr int kDzTile = 64;

__global__ void __launch_bounds__(256) dlogits_kernel(const DlogitParams p) {
  __shared__ uint16_t tile[kDzTile][kDzTile + 2];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int r0 = blockIdx.y * kDzTile, c0 = blockIdx.x * kDzTile;
  const int64_t n_valid = p.hdr->n_valid;
  float coef;
  if (n_valid == 0) {
    coef = 0.f;
  } else {
    coef = p.reduction == FLCE_REDUCTION_MEAN ? p.grad_scale / static_cast<float>(n_valid) : p.grad_scale;
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int lr = ty + 16 * k;
    const int r = r0 + lr;
    const int c = c0 + tx * 4;
    float d[4] = {0.f, 0.f, 0.f, 0.f};
    if (r < p.rows) {
      const int64_t y = p.labels[r];
      const bool valid = y != p.ignore_index;
      const float ci = valid ? coef : 0.f;
      const float lse = p.lse[r];
      const float* srow = p.s + static_cast<int64_t>(r) * p.lds;
      if (c + 3 < p.vocab) {
        const float4 v = *reinterpret_cast<const float4*>(srow + c);
        const float sv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          float q = ci * (__expf(sv[j] - lse) - ((c + j) == y ? 1.f : 0.f));
          if (p.softcap > 0.f) {
            const float u = sv[j] * p.inv_softcap;
            q *= (1.f - u * u);
          }
          d[j] = q;
        }
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (c + j < p.vocab) {
            const float sv = srow[c + j];
            float q = ci * (__expf(sv - lse) - ((c + j) == y ? 1.f : 0.f));
            if (p.softcap > 0.f) {
              const float u = sv * p.inv_softcap;
              q *= (1.f - u * u);
            }
            d[j] = q;
          }
        }
      }
    }
    uint16_t b[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      b[j] = float_to_bf16_bits(d[j]);
      tile[lr][tx * 4 + j] = b[j];
    }
    if (p.dz && r < p.rows && c < p.vocab) {
      uint16_t* drow = p.dz + static_cast<int64_t>(r) * p.ldd;
      if (c + 3 < p.vocab) {
        uint2 pk;
        pk.x = static_cast<uint32_t>(b[0]) | (static_cast<uint32_t>(b[1]) << 16);
        pk.y = static_cast<uint32_t>(b[2]) | (static_cast<uint32_t>(b[3]) << 16);
        *reinterpret_cast<uint2*>(drow + c) = pk;
      } else {
        for (int j = 0; j < 4; ++j)
          if (c + j < p.vocab) drow[c + j] = b[j];
      }
    }
  }
  if (!p.dzt) return;
  __syncthreads();
  // dzt [vocab][ldt]: row = vocab column, contiguous along the chunk rows.
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int lc = ty + 16 * k;
    const int c = c0 + lc;
    const int r = r0 + tx * 4;
    if (c < p.vocab && r < p.rows) {
      uint16_t* trow = p.dzt + static_cast<int64_t>(c) * p.ldt;
      if (r + 3 < p.rows) {
        uint2 pk;
        pk.x = static_cast<uint32_t>(tile[tx * 4 + 0][lc]) | (static_cast<uint32_t>(tile[tx * 4 + 1][lc]) << 16);
        pk.y = static_cast<uint32_t>(tile[tx * 4 + 2][lc]) | (static_cast<uint32_t>(tile[tx * 4 + 3][lc]) << 16);
        *reinterpret_cast<uint2*>(trow + r) = pk;
      } else {
        for (int j = 0; j < 4; ++j)
          if (r + j < p.rows) trow[r + j] = tile[tx * 4 + j][lc];
      }
    }
  }
}

// Product path (no transposed copy): plain streaming over the rows. A block
// covers 8192 columns of one row; thread t handles four 8-column pieces
// 2048 i + 8 t (each piece: 32 B of s read, 16 B of dz written, contiguous
// across the block), so the per-row setup is paid once per 32 columns.
// exp(s - lse) is 2^(s log2 e - lse log2 e) on the special-function unit.
// HALF: the forward stored s - gmax in fp16 (s16) with gmax per 32-column
// group; the eight columns of a piece lie in one group.
template <bool CAP, bool HALF>
__device__ __forceinline__ void dlogits_piece(const DlogitParams& p, const float* srow, const uint16_t* s16row,
                                              const float* grow, uint16_t* drow, int c, float ci, float lse_l2e,
                                              int label_local) {
  float sv[8];
  const bool full = c + 8 <= p.vocab;
  if (HALF) {
    const float gm = grow[c >> 5];
    if (full) {
      const uint4 a = *reinterpret_cast<const uint4*>(s16row + c);
      const uint32_t w4[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w4[j]));
        sv[2 * j] = f.x + gm;
        sv[2 * j + 1] = f.y + gm;
      }
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j)
        sv[j] = (c + j < p.vocab) ? __half2float(__ushort_as_half(s16row[c + j])) + gm : 0.f;
    }
  } else if (full) {
    const float4 a = *reinterpret_cast<const float4*>(srow + c);
    const float4 b = *reinterpret_cast<const float4*>(srow + c + 4);
    sv[0] = a.x; sv[1] = a.y; sv[2] = a.z; sv[3] = a.w;
    sv[4] = b.x; sv[5] = b.y; sv[6] = b.z; sv[7] = b.w;
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j) sv[j] = (c + j < p.vocab) ? srow[c + j] : 0.f;
  }
  uint32_t w[4];
#pragma unroll
  for (int j = 0; j < 8; j += 2) {
    float q0 = ex2_approx(fmaf(sv[j], 1.4426950408889634f, -lse_l2e)) - (j == label_local ? 1.f : 0.f);
    float q1 = ex2_approx(fmaf(sv[j + 1], 1.4426950408889634f, -lse_l2e)) - (j + 1 == label_local ? 1.f : 0.f);
    if (CAP) {
      const float u0 = sv[j] * p.inv_softcap, u1 = sv[j + 1] * p.inv_softcap;
      q0 *= (1.f - u0 * u0);
      q1 *= (1.f - u1 * u1);
    }
    w[j / 2] = static_cast<uint32_t>(float_to_bf16_bits(ci * q0)) |
               (static_cast<uint32_t>(float_to_bf16_bits(ci * q1)) << 16);
  }
  if (full) {
    *reinterpret_cast<uint4*>(drow + c) = make_uint4(w[0], w[1], w[2], w[3]);
  } else {
    for (int j = 0; j < 8; ++j)
      if (c + j < p.vocab) drow[c + j] = static_cast<uint16_t>(w[j / 2] >> (16 * (j & 1)));
  }
}

template <bool HALF>
__global__ void __launch_bounds__(256) dlogits_rows_kernel(const DlogitParams p) {
  const int r = blockIdx.y;
  const int c_base = blockIdx.x * 8192 + threadIdx.x * 8;
  if (c_base >= p.vocab) return;
  const int64_t n_valid = p.hdr->n_valid;
  const int64_t y = p.labels[r];
  float ci = 0.f;
  if (y != p.ignore_index && n_valid > 0)
    ci = p.reduction == FLCE_REDUCTION_MEAN ? p.grad_scale / static_cast<float>(n_valid) : p.grad_scale;
  const float lse_l2e = p.lse[r] * 1.4426950408889634f;
  const float* srow = HALF ? nullptr : p.s + static_cast<int64_t>(r) * p.lds;
  const uint16_t* s16row = HALF ? p.s16 + static_cast<int64_t>(r) * p.lds : nullptr;
  const float* grow = HALF ? p.gmax + static_cast<int64_t>(r) * p.ldg : nullptr;
  uint16_t* drow = p.dz + static_cast<int64_t>(r) * p.ldd;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int c = c_base + i * 2048;
    if (c >= p.vocab) break;
    const int64_t dl = y - p.label_offset - c;
    const int label_local = (dl >= 0 && dl < 8) ? static_cast<int>(dl) : -1;
    if (p.softcap > 0.f)
      dlogits_piece<true, HALF>(p, srow, s16row, grow, drow, c, ci, lse_l2e, label_local);
    else
      dlogits_piece<false, HALF>(p, srow, s16row, grow, drow, c, ci, lse_l2e, label_local);
  }
}

// fp32-operand path: dz and dz^T in fp32 (64x64 tiles, transposed through
// shared memory as in the bf16 kernel above).
__global__ void __launch_bounds__(256) dlogits_f32_kernel(const DlogitParams p) {
  __shared__ float tile[kDzTile][kDzTile + 1];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int r0 = blockIdx.y * kDzTile, c0 = blockIdx.x * kDzTile;
  const int64_t n_valid = p.hdr->n_valid;
  const float coef = n_valid == 0 ? 0.f
                                  : (p.reduction == FLCE_REDUCTION_MEAN ? p.grad_scale / static_cast<float>(n_valid)
                                                                        : p.grad_scale);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int lr = ty + 16 * k;
    const int r = r0 + lr;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int c = c0 + tx * 4 + j;
      float q = 0.f;
      if (r < p.rows && c < p.vocab) {
        const int64_t y = p.labels[r];
        const float ci = y != p.ignore_index ? coef : 0.f;
        const float sv = p.s[static_cast<int64_t>(r) * p.lds + c];
        q = ci * (__expf(sv - p.lse[r]) - (c == y ? 1.f : 0.f));
        if (p.softcap > 0.f) {
          const float u = sv * p.inv_softcap;
          q *= (1.f - u * u);
        }
        if (p.dz32) {
          if (p.dz32_lo) {
            float hi, lo;
            split_tf32(q, hi, lo);
            p.dz32[static_cast<int64_t>(r) * p.ldd + c] = hi;
            p.dz32_lo[static_cast<int64_t>(r) * p.ldd + c] = lo;
          } else {
            p.dz32[static_cast<int64_t>(r) * p.ldd + c] = q;
          }
        }
      }
      tile[lr][tx * 4 + j] = q;
    }
  }
  if (!p.dzt32) return;
  __syncthreads();
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int lc = ty + 16 * k;
    const int c = c0 + lc;
    if (c >= p.vocab) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int r = r0 + tx * 4 + j;
      if (r >= p.rows) continue;
      const float q = tile[tx * 4 + j][lc];
      if (p.dzt32_lo) {
        float hi, lo;
        split_tf32(q, hi, lo);
        p.dzt32[static_cast<int64_t>(c) * p.ldt + r] = hi;
        p.dzt32_lo[static_cast<int64_t>(c) * p.ldt + r] = lo;
      } else {
        p.dzt32[static_cast<int64_t>(c) * p.ldt + r] = q;
      }
    }
  }
}

cudaError_t launch_dlogits(const DlogitParams& p, cudaStream_t s) {
  if (p.rows <= 0 || p.vocab <= 0) return cudaSuccess;
  if (p.dz32 != nullptr || p.dzt32 != nullptr) {
    dim3 grid((p.vocab + kDzTile - 1) / kDzTile, (p.rows + kDzTile - 1) / kDzTile);
    dlogits_f32_kernel<<<grid, 256, 0, s>>>(p);
    return cudaGetLastError();
  }
  if (p.dzt == nullptr && p.dz != nullptr) {
    dim3 grid((p.vocab + 8191) / 8192, p.rows);
    if (p.s16 != nullptr)
      dlogits_rows_kernel<true><<<grid, 256, 0, s>>>(p);
    else
      dlogits_rows_kernel<false><<<grid, 256, 0, s>>>(p);
    return cudaGetLastError();
  }
  dim3 grid((p.vocab + kDzTile - 1) / kDzTile, (p.rows + kDzTile - 1) / kDzTile);
  dlogits_kernel<<<grid, 256, 0, s>>>(p);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ transpose
__global__ void __launch_bounds__(256) transpose_bf16_kernel(const uint16_t* __restrict__ in, int64_t ldi,
                                                             int rows, int cols, uint16_t* __restrict__ out,
                                                             int64_t ldo) {
  __shared__ uint16_t tile[64][66];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int r0 = blockIdx.y * 64, c0 = blockIdx.x * 64;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int lr = ty + 16 * k;
    const int r = r0 + lr;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int c = c0 + tx * 4 + j;
      tile[lr][tx * 4 + j] = (r < rows && c < cols) ? in[static_cast<int64_t>(r) * ldi + c] : 0;
    }
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int lc = ty + 16 * k;
    const int c = c0 + lc;
    if (c >= cols) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int r = r0 + tx * 4 + j;
      if (r < rows) out[static_cast<int64_t>(c) * ldo + r] = tile[tx * 4 + j][lc];
    }
  }
}

cudaError_t launch_transpose_bf16(const uint16_t* in, int64_t ldi, int rows, int cols, uint16_t* out, int64_t ldo,
                                  cudaStream_t s) {
  if (rows <= 0 || cols <= 0) return cudaSuccess;
  dim3 grid((cols + 63) / 64, (rows + 63) / 64);
  transpose_bf16_kernel<<<grid, 256, 0, s>>>(in, ldi, rows, cols, out, ldo);
  return cudaGetLastError();
}

__global__ void __launch_bounds__(256) transpose_f32_kernel(const float* __restrict__ in, int64_t ldi, int rows,
                                                            int cols, float* __restrict__ out, int64_t ldo,
                                                            float* __restrict__ out_lo) {
  __shared__ float tile[64][65];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int r0 = blockIdx.y * 64, c0 = blockIdx.x * 64;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int lr = ty + 16 * k;
    const int r = r0 + lr;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int c = c0 + tx * 4 + j;
      tile[lr][tx * 4 + j] = (r < rows && c < cols) ? in[static_cast<int64_t>(r) * ldi + c] : 0.f;
    }
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int lc = ty + 16 * k;
    const int c = c0 + lc;
    if (c >= cols) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int r = r0 + tx * 4 + j;
      if (r >= rows) continue;
      const float v = tile[tx * 4 + j][lc];
      if (out_lo) {
        float hi, lo;
        split_tf32(v, hi, lo);
        out[static_cast<int64_t>(c) * ldo + r] = hi;
        out_lo[static_cast<int64_t>(c) * ldo + r] = lo;
      } else {
        out[static_cast<int64_t>(c) * ldo + r] = v;
      }
    }
  }
}

cudaError_t launch_transpose_f32(const float* in, int64_t ldi, int rows, int cols, float* out, int64_t ldo,
                                 cudaStream_t s, float* out_lo) {
  if (rows <= 0 || cols <= 0) return cudaSuccess;
  dim3 grid((cols + 63) / 64, (rows + 63) / 64);
  transpose_f32_kernel<<<grid, 256, 0, s>>>(in, ldi, rows, cols, out, ldo, out_lo);
  return cudaGetLastError();
}

// hi [rows][ldo], lo [rows][ldo] = the tf32 split of in [rows][ldi] (cols columns).
__global__ void __launch_bounds__(256) split_f32_kernel(const float* __restrict__ in, int64_t ldi, int rows, int cols,
                                                        float* __restrict__ hi, float* __restrict__ lo, int64_t ldo) {
  const int r = blockIdx.y;
  for (int c = blockIdx.x * blockDim.x + threadIdx.x; c < cols; c += gridDim.x * blockDim.x) {
    float h, l;
    split_tf32(in[static_cast<int64_t>(r) * ldi + c], h, l);
    hi[static_cast<int64_t>(r) * ldo + c] = h;
    lo[static_cast<int64_t>(r) * ldo + c] = l;
  }
}

cudaError_t launch_split_f32(const float* in, int64_t ldi, int rows, int cols, float* hi, float* lo, int64_t ldo,
                             cudaStream_t s) {
  if (rows <= 0 || cols <= 0) return cudaSuccess;
  for (int r0 = 0; r0 < rows; r0 += 65535) {  // grid.y per launch stays within its limit
    const int nr = rows - r0 < 65535 ? rows - r0 : 65535;
    dim3 grid((cols + 255) / 256 < 8 ? (cols + 255) / 256 : 8, nr);
    split_f32_kernel<<<grid, 256, 0, s>>>(in + static_cast<int64_t>(r0) * ldi, ldi, nr, cols,
                                           hi + static_cast<int64_t>(r0) * ldo, lo + static_cast<int64_t>(r0) * ldo,
                                           ldo);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// ------------------------------------------------------------------ convert
__global__ void __launch_bounds__(256) f32_to_bf16_kernel(const float* __restrict__ in, uint16_t* __restrict__ out,
                                                          int64_t n) {
  const int64_t i = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) * 4;
  if (i + 4 <= n) {
    const float4 v = *reinterpret_cast<const float4*>(in + i);
    uint2 pk;
    pk.x = static_cast<uint32_t>(float_to_bf16_bits(v.x)) | (static_cast<uint32_t>(float_to_bf16_bits(v.y)) << 16);
    pk.y = static_cast<uint32_t>(float_to_bf16_bits(v.z)) | (static_cast<uint32_t>(float_to_bf16_bits(v.w)) << 16);
    *reinterpret_cast<uint2*>(out + i) = pk;
  } else {
    for (int64_t j = i; j < n; ++j) out[j] = float_to_bf16_bits(in[j]);
  }
}

cudaError_t launch_f32_to_bf16(const float* in, uint16_t* out, int64_t n, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  const int64_t threads = (n + 3) / 4;
  f32_to_bf16_kernel<<<static_cast<unsigned>((threads + 255) / 256), 256, 0, s>>>(in, out, n);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ scale
// y = scale * x converted to y's type: a streaming pass, 8 elements per thread
// and step (two or one 16-byte accesses), grid-stride over a persistent grid.
__device__ __forceinline__ void load8(const float* p, float v[8]) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  const float4 b = *reinterpret_cast<const float4*>(p + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void load8(const uint16_t* p, float v[8]) {
  const uint4 a = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    v[2 * j] = __uint_as_float(w[j] << 16);
    v[2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
  }
}
__device__ __forceinline__ void store8(float* p, const float v[8]) {
  *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  *reinterpret_cast<float4*>(p + 4) = make_float4(v[4], v[5], v[6], v[7]);
}
__device__ __forceinline__ void store8(uint16_t* p, const float v[8]) {
  uint4 a;
  a.x = static_cast<uint32_t>(float_to_bf16_bits(v[0])) | (static_cast<uint32_t>(float_to_bf16_bits(v[1])) << 16);
  a.y = static_cast<uint32_t>(float_to_bf16_bits(v[2])) | (static_cast<uint32_t>(float_to_bf16_bits(v[3])) << 16);
  a.z = static_cast<uint32_t>(float_to_bf16_bits(v[4])) | (static_cast<uint32_t>(float_to_bf16_bits(v[5])) << 16);
  a.w = static_cast<uint32_t>(float_to_bf16_bits(v[6])) | (static_cast<uint32_t>(float_to_bf16_bits(v[7])) << 16);
  *reinterpret_cast<uint4*>(p) = a;
}
__device__ __forceinline__ float load1(const float* p) { return *p; }
__device__ __forceinline__ float load1(const uint16_t* p) { return bf16_bits_to_float(*p); }
__device__ __forceinline__ void store1(float* p, float v) { *p = v; }
__device__ __forceinline__ void store1(uint16_t* p, float v) { *p = float_to_bf16_bits(v); }

// VEC: both pointers 16-byte aligned, so every 8-element group is one or two
// aligned vector accesses; otherwise element by element.
template <typename TI, typename TO, bool VEC>
__global__ void __launch_bounds__(256) scale_convert_kernel(const TI* x, TO* y, int64_t n, const float* scale) {
  const float c = scale ? *scale : 1.0f;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (VEC) {
    const int64_t groups = n / 8;
    const TI* xp = x + tid * 8;
    TO* yp = y + tid * 8;
    for (int64_t g = tid; g < groups; g += stride, xp += stride * 8, yp += stride * 8) {
      float v[8];
      load8(xp, v);
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] *= c;
      store8(yp, v);
    }
    for (int64_t i = groups * 8 + tid; i < n; i += stride) store1(y + i, c * load1(x + i));
  } else {
    for (int64_t i = tid; i < n; i += stride) store1(y + i, c * load1(x + i));
  }
}

template <typename TI, typename TO>
cudaError_t launch_scale_typed(const void* x, void* y, int64_t n, const float* scale, int sms, cudaStream_t s) {
  const int64_t groups = (n + 7) / 8;
  const int64_t want = (groups + 255) / 256;
  const unsigned blocks = static_cast<unsigned>(want < 4LL * sms ? want : 4LL * sms);
  const bool vec = (reinterpret_cast<uintptr_t>(x) % 16 == 0) && (reinterpret_cast<uintptr_t>(y) % 16 == 0);
  if (vec)
    scale_convert_kernel<TI, TO, true><<<blocks, 256, 0, s>>>(static_cast<const TI*>(x), static_cast<TO*>(y), n, scale);
  else
    scale_convert_kernel<TI, TO, false><<<blocks, 256, 0, s>>>(static_cast<const TI*>(x), static_cast<TO*>(y), n, scale);
  return cudaGetLastError();
}

cudaError_t launch_scale_convert(const void* x, bool x_f32, void* y, bool y_f32, int64_t n, const float* scale,
                                 int sms, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  if (x_f32 && y_f32) return launch_scale_typed<float, float>(x, y, n, scale, sms, s);
  if (x_f32) return launch_scale_typed<float, uint16_t>(x, y, n, scale, sms, s);
  if (y_f32) return launch_scale_typed<uint16_t, float>(x, y, n, scale, sms, s);
  return launch_scale_typed<uint16_t, uint16_t>(x, y, n, scale, sms, s);
}

// ------------------------------------------------------------------ finish
__global__ void finish_kernel(const Header* hdr, int reduction, float* loss, float* token_accuracy) {
  const int64_t nv = hdr->n_valid;
  float l = 0.f, a = 0.f;
  if (nv > 0) {
    l = reduction == FLCE_REDUCTION_MEAN ? static_cast<float>(hdr->loss_sum / static_cast<double>(nv))
                                         : static_cast<float>(hdr->loss_sum);
    a = static_cast<float>(static_cast<double>(hdr->correct) / static_cast<double>(nv));
  }
  if (loss) *loss = l;
  if (token_accuracy) *token_accuracy = a;
}

cudaError_t launch_finish(const Header* hdr, int reduction, float* loss, float* token_accuracy, cudaStream_t s) {
  finish_kernel<<<1, 1, 0, s>>>(hdr, reduction, loss, token_accuracy);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ debug SIMT GEMM
// 64x64 tile per 256-thread block, 4x4 outputs per thread, fp32 FMA.
template <int MODE>
__global__ void __launch_bounds__(256) gemm_simt_kernel(const uint16_t* __restrict__ A, int64_t lda,
                                                        const uint16_t* __restrict__ B, int64_t ldb,
                                                        const GemmParams p) {
  __shared__ float As[32][65];
  __shared__ float Bs[32][65];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  for (int k0 = 0; k0 < p.K; k0 += 32) {
    for (int e = threadIdx.x; e < 64 * 32; e += 256) {
      const int r = e >> 5, c = e & 31;
      const int gm = m0 + r, gn = n0 + r, gk = k0 + c;
      As[c][r] = (gm < p.M_valid && gk < p.K)
                     ? bf16_bits_to_float(A[static_cast<int64_t>(p.a_row0 + gm) * lda + gk])
                     : 0.f;
      Bs[c][r] = (gn < p.N && gk < p.K) ? bf16_bits_to_float(B[static_cast<int64_t>(p.b_row0 + gn) * ldb + gk])
                                       : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < 32; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int gm = m0 + ty * 4 + i;
    if (gm >= p.M_valid) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int gn = n0 + tx * 4 + j;
      if (gn >= p.N_valid) continue;
      const float v = acc[i][j] * p.alpha;
      if (MODE == EPI_STATS || MODE == EPI_STATS_STORE) {
        p.zbuf[static_cast<int64_t>(gm) * p.ldz + gn] = v;
      } else if (MODE == EPI_BF16) {
        static_cast<uint16_t*>(p.out)[static_cast<int64_t>(gm) * p.ldo + gn] = float_to_bf16_bits(v);
      } else {
        static_cast<float*>(p.out)[static_cast<int64_t>(gm) * p.ldo + gn] += v;
      }
    }
  }
}

cudaError_t launch_gemm_simt(int mode, const void* A, int64_t lda, const void* B, int64_t ldb, const GemmParams& p,
                             cudaStream_t s) {
  if (p.M_valid <= 0 || p.N <= 0) return cudaSuccess;
  dim3 grid((p.N + 63) / 64, (p.M_valid + 63) / 64);
  const uint16_t* a = static_cast<const uint16_t*>(A);
  const uint16_t* b = static_cast<const uint16_t*>(B);
  switch (mode) {
    case EPI_STATS:
    case EPI_STATS_STORE: gemm_simt_kernel<EPI_STATS><<<grid, 256, 0, s>>>(a, lda, b, ldb, p); break;
    case EPI_BF16: gemm_simt_kernel<EPI_BF16><<<grid, 256, 0, s>>>(a, lda, b, ldb, p); break;
    case EPI_ACC_F32: gemm_simt_kernel<EPI_ACC_F32><<<grid, 256, 0, s>>>(a, lda, b, ldb, p); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

// Statistics of one 256-column vocab tile per thread-row from the logits the
// SIMT GEMM stored (z = m h W^T in zbuf); optionally overwrites them with the
// capped logits s for the dlogits pass.
__global__ void __launch_bounds__(128) stats_from_z_kernel(const GemmParams p, int rows, int store) {
  const int nb = blockIdx.x;
  const int row = blockIdx.y * 128 + threadIdx.x;
  if (row >= rows) return;
  const int n0 = nb * kVTile;
  const int64_t label = p.labels[row];
  const bool has_label = label != p.ignore_index && label >= n0 && label < n0 + kVTile;
  float* zrow = p.zbuf + static_cast<int64_t>(row) * p.ldz;
  RowStats st;
  row_stats_init(st, n0);
  for (int c = 0; c < kVTile / 32; ++c) {
    float s[32];
    const int col0 = n0 + c * 32;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const bool in = col0 + j < p.N_valid;
      s[j] = cap_logit(in ? zrow[col0 + j] : 0.f, p.softcap, p.inv_softcap, in);
    }
    if (store) {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (col0 + j < p.N_valid) zrow[col0 + j] = s[j];
    }
    row_stats_update32(st, s, col0, has_label ? label : -1);
  }
  const int64_t o = static_cast<int64_t>(nb) * p.ldp + row;
  p.part_max[o] = st.mx;
  p.part_sum[o] = st.sum;
  p.part_idx[o] = st.arg;
  if (has_label) p.tgt[row] = st.tgt;
}

cudaError_t launch_stats_from_z(const GemmParams& p, int rows, bool store, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  dim3 grid(p.n_tiles, (rows + 127) / 128);
  stats_from_z_kernel<<<grid, 128, 0, s>>>(p, rows, store ? 1 : 0);
  return cudaGetLastError();
}

}  // namespace flce
