// Per-row forward statistics shared by the tensor-core GEMM epilogue and the
// debug path: softcap, running max / sum of exponentials, argmax and the
// label's capped logit over one 256-column vocab tile of one row.
#pragma once

#include <math.h>
#include <stdint.h>

#include "flce_device.cuh"

namespace flce {

// Capped logit (Liger-Kernel "Muse Glimmer" page, Details / Softcap): the fused
// path sees z = m (h W^T) with m applied as the GEMM scale, and caps it as
// T tanh(z / T). T = 0 leaves z unchanged. Columns at or past V get -inf so
// they drop out of the max, the sum and the argmax.
__device__ __forceinline__ float cap_logit(float z, float softcap, float inv_softcap, bool in_vocab) {
  const float s = softcap > 0.f ? softcap * tanhf(z * inv_softcap) : z;
  return in_vocab ? s : -INFINITY;
}

// Capped logits of one 32-column group from the fp32 accumulator bits r:
// s = T tanh(u / T) with u = alpha * acc (the softcap of the Liger-Kernel "Muse
// Glimmer" page, Details / Softcap).
// Where |u / T| < 1/2 for every value the warp holds in this group (always on
// the heads this library is measured on: |z| / T stays below 0.2 there), tanh
// comes from its odd Taylor-like form tanh(x) = x P(x^2), with P of degree 5
// fitted here by least squares on Chebyshev nodes of [0, 1/4] to tanh(x) / x
// (constant term 1), so s = u P((u / T)^2): packed FMAs only, within 1.2 ulp of
// the exact T tanh(u / T) in fp32 (a tighter bound than T * tanhf(u / T), whose
// own rounding steps allow about 3 ulp). Any larger argument in the group sends
// the whole warp to T * tanhf(u / T). NaN stays NaN either way.
__device__ __forceinline__ void softcap32(float (&s)[32], const uint32_t (&r)[32], float alpha, float T,
                                          float invT) {
  const uint64_t al2 = f2_pack(alpha, alpha);
  const uint64_t it2 = f2_pack(invT, invT);
  const uint64_t p5 = f2_pack(-0.0069470275193452835f, -0.0069470275193452835f);
  const uint64_t p4 = f2_pack(0.021472735330462456f, 0.021472735330462456f);
  const uint64_t p3 = f2_pack(-0.05393379181623459f, -0.05393379181623459f);
  const uint64_t p2 = f2_pack(0.1333322674036026f, 0.1333322674036026f);
  const uint64_t p1 = f2_pack(-0.3333333134651184f, -0.3333333134651184f);
  const uint64_t p0 = f2_pack(1.f, 1.f);
  float xmax = 0.f;
#pragma unroll
  for (int j = 0; j < 32; j += 2) {
    const uint64_t u = f2_mul(f2_pack(__uint_as_float(r[j]), __uint_as_float(r[j + 1])), al2);
    const uint64_t x = f2_mul(u, it2);
    float x0, x1;
    f2_unpack(x, x0, x1);
    xmax = max3f(xmax, fabsf(x0), fabsf(x1));
    const uint64_t w = f2_mul(x, x);
    uint64_t q = f2_fma(p5, w, p4);
    q = f2_fma(q, w, p3);
    q = f2_fma(q, w, p2);
    q = f2_fma(q, w, p1);
    q = f2_fma(q, w, p0);
    f2_unpack(f2_mul(u, q), s[j], s[j + 1]);
  }
  if (!__all_sync(0xffffffffu, xmax < 0.5f)) {
#pragma unroll
    for (int j = 0; j < 32; ++j) s[j] = T * tanhf(__uint_as_float(r[j]) * alpha * invT);
  }
}

struct RowStats {
  float mx;    // running max of s over the tile so far (= value at the argmax)
  float sum;   // sum of exp(s - mx)
  int arg;     // vocab index of the first maximum
  float tgt;   // s at the label column, when the label falls in this tile
  bool first;  // (no-argmax form) s at the label is above every earlier column of the tile
};

__device__ __forceinline__ void row_stats_init(RowStats& st, int col0) {
  st.mx = -INFINITY;
  st.sum = 0.f;
  st.arg = col0;
  st.tgt = 0.f;
  st.first = false;
}

// The running sum of exponentials over 32 columns, after the running max has
// taken in this group: 2^(s log2 e - mx log2 e), one packed FMA per two columns
// and four running sums (two packed) in the order of four scalar ones.
__device__ __forceinline__ void row_sum_exp32(RowStats& st, const float (&s)[32]) {
  const float mx_l2e = st.mx * 1.4426950408889634f;
  const uint64_t l2e2 = f2_pack(1.4426950408889634f, 1.4426950408889634f);
  const uint64_t nmx2 = f2_pack(-mx_l2e, -mx_l2e);
  uint64_t a01 = f2_pack(0.f, 0.f), a23 = a01;
#pragma unroll
  for (int j = 0; j < 32; j += 4) {
    float x0, x1, x2, x3;
    f2_unpack(f2_fma(f2_pack(s[j], s[j + 1]), l2e2, nmx2), x0, x1);
    f2_unpack(f2_fma(f2_pack(s[j + 2], s[j + 3]), l2e2, nmx2), x2, x3);
    a01 = f2_add(a01, f2_pack(ex2_approx(x0), ex2_approx(x1)));
    a23 = f2_add(a23, f2_pack(ex2_approx(x2), ex2_approx(x3)));
  }
  float a0, a1, a2, a3;
  f2_unpack(a01, a0, a1);
  f2_unpack(a23, a2, a3);
  st.sum += (a0 + a1) + (a2 + a3);
}

// s at column d of the group, without a dynamically indexed (local-memory)
// array: a predicated select per column.
__device__ __forceinline__ float select_col32(const float (&s)[32], int d, float t) {
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const bool hit = (j == d);
    asm("{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %2, 0;\n\t@q mov.f32 %0, %1;\n\t}\n"
        : "+f"(t)
        : "f"(s[j]), "r"(static_cast<uint32_t>(hit)));
  }
  return t;
}

// Folds 32 consecutive columns col0 .. col0+31 of one row into `st`, and
// returns the largest of the 32 values.
// The group's max comes from the maxima of its four 8-column quarters (trees
// of three-input maxima). Only where it raises the running max, that is where
// the tile gets a new first maximum, is its column looked up: the first
// quarter whose max equals it, then the first column of that quarter that
// does. Earlier columns win every tie, and against earlier groups the running
// max is replaced only on a strict increase, so the index is the lowest one
// holding the tile's maximum. exp(s - mx) is computed as 2^(s log2 e - mx log2 e).
__device__ __forceinline__ float row_stats_update32(RowStats& st, const float (&s)[32], int col0,
                                                    int64_t label) {
  float q[4];
#pragma unroll
  for (int k = 0; k < 4; ++k)
    q[k] = max3f(max3f(s[8 * k], s[8 * k + 1], s[8 * k + 2]), max3f(s[8 * k + 3], s[8 * k + 4], s[8 * k + 5]),
                 fmaxf(s[8 * k + 6], s[8 * k + 7]));
  const float cm = max3f(q[0], q[1], fmaxf(q[2], q[3]));
  if (cm > st.mx) {
    st.sum *= ex2_approx((st.mx - cm) * 1.4426950408889634f);
    st.mx = cm;
    const bool in0 = q[0] == cm, in1 = q[1] == cm, in2 = q[2] == cm;
    float v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = in0 ? s[j] : in1 ? s[8 + j] : in2 ? s[16 + j] : s[24 + j];
    int jj = 7;
#pragma unroll
    for (int j = 6; j >= 0; --j) jj = v[j] == cm ? j : jj;
    st.arg = col0 + (in0 ? 0 : in1 ? 8 : in2 ? 16 : 24) + jj;
  }
  row_sum_exp32(st, s);
  // the label's logit, taken only by rows whose label is in this group
  const int64_t d64 = label - col0;
  if (d64 >= 0 && d64 < 32) st.tgt = select_col32(s, static_cast<int>(d64), st.tgt);
  return cm;
}

// The same fold without the argmax, for calls that return token accuracy but
// not the predicted tokens: the group's max by a tree of three-input maxima,
// and, in the group holding the row's label (column d of the group, else d
// outside 0..31), whether the label's logit lies strictly above every earlier
// column of the tile. The label is the row's first maximum exactly when that
// holds, the logit equals the tile's max, and no earlier tile reaches it.
// The sums and the running max take the same steps as row_stats_update32.
__device__ __forceinline__ float row_stats_update32_noarg(RowStats& st, const float (&s)[32], int d) {
  float m[11];
#pragma unroll
  for (int k = 0; k < 10; ++k) m[k] = max3f(s[3 * k], s[3 * k + 1], s[3 * k + 2]);
  m[10] = fmaxf(s[30], s[31]);
  const float cm = fmaxf(max3f(max3f(m[0], m[1], m[2]), max3f(m[3], m[4], m[5]), max3f(m[6], m[7], m[8])),
                         fmaxf(m[9], m[10]));
  const float prev = st.mx;  // max of the tile's earlier columns
  if (cm > st.mx) {
    st.sum *= ex2_approx((st.mx - cm) * 1.4426950408889634f);
    st.mx = cm;
  }
  row_sum_exp32(st, s);
  if (d >= 0 && d < 32) {
    const float t = select_col32(s, d, st.tgt);
    bool first = prev < t;
#pragma unroll
    for (int j = 0; j < 31; ++j) first = first && !(j < d && !(s[j] < t));
    st.tgt = t;
    st.first = first;
  }
  return cm;
}

}  // namespace flce
