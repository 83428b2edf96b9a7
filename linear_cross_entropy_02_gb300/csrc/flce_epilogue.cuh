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

struct RowStats {
  float mx;    // running max of s over the tile so far (= value at the argmax)
  float sum;   // sum of exp(s - mx)
  int arg;     // vocab index of the first maximum
  float tgt;   // s at the label column, when the label falls in this tile
};

__device__ __forceinline__ void row_stats_init(RowStats& st, int col0) {
  st.mx = -INFINITY;
  st.sum = 0.f;
  st.arg = col0;
  st.tgt = 0.f;
}

// One level of the adjacent-pairs argmax tree: slot j takes the larger of slots
// 2j and 2j+1 (which cover lower and higher columns); equal values keep the left.
template <int W>
__device__ __forceinline__ void pair_level(float (&v)[16], int (&ix)[16]) {
#pragma unroll
  for (int j = 0; j < W; ++j) {
    const bool right = v[2 * j + 1] > v[2 * j];
    v[j] = right ? v[2 * j + 1] : v[2 * j];
    ix[j] = right ? ix[2 * j + 1] : ix[2 * j];
  }
}

// Folds 32 consecutive columns col0 .. col0+31 of one row into `st`, and
// returns the largest of the 32 values.
// Argmax over the 32 by a tree of adjacent pairs, so the left operand always
// holds the lower columns and a strict comparison keeps the lowest index on
// ties; against earlier columns the running max is also replaced only on a
// strict increase. exp(s - mx) is computed as 2^(s log2 e - mx log2 e).
__device__ __forceinline__ float row_stats_update32(RowStats& st, const float (&s)[32], int col0,
                                                    int64_t label) {
  float v[16];
  int ix[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const bool right = s[2 * j + 1] > s[2 * j];
    v[j] = right ? s[2 * j + 1] : s[2 * j];
    ix[j] = right ? 2 * j + 1 : 2 * j;
  }
  pair_level<8>(v, ix);
  pair_level<4>(v, ix);
  pair_level<2>(v, ix);
  pair_level<1>(v, ix);
  const float cm = v[0];
  if (cm > st.mx) {
    st.sum *= ex2_approx((st.mx - cm) * 1.4426950408889634f);
    st.mx = cm;
    st.arg = col0 + ix[0];
  }
  const float mx_l2e = st.mx * 1.4426950408889634f;
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
  for (int j = 0; j < 32; j += 4) {
    a0 += ex2_approx(fmaf(s[j + 0], 1.4426950408889634f, -mx_l2e));
    a1 += ex2_approx(fmaf(s[j + 1], 1.4426950408889634f, -mx_l2e));
    a2 += ex2_approx(fmaf(s[j + 2], 1.4426950408889634f, -mx_l2e));
    a3 += ex2_approx(fmaf(s[j + 3], 1.4426950408889634f, -mx_l2e));
  }
  st.sum += (a0 + a1) + (a2 + a3);
  // Label gather without a dynamically indexed (local-memory) array: a
  // predicated select per column, taken only by rows whose label is here.
  const int64_t d64 = label - col0;
  if (d64 >= 0 && d64 < 32) {
    const int d = static_cast<int>(d64);
    float t = st.tgt;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const bool hit = (j == d);
      asm("{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %2, 0;\n\t@q mov.f32 %0, %1;\n\t}\n"
          : "+f"(t)
          : "f"(s[j]), "r"(static_cast<uint32_t>(hit)));
    }
    st.tgt = t;
  }
  return cm;
}

}  // namespace flce
