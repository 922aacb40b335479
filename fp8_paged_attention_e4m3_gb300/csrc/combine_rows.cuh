// The combine of one unit (output row r of sequence b, KV head h, 64-wide
// slice of d) over the FP32 partition states, by a group of 256 threads:
//     M   = max_p m_p  (live partitions: l_p > 0)
//     w_p = 2^(m_p - M)
//     out = (sum_p w_p O_p) / (sum_p w_p l_p) * s_V * 2^8   -> FP16 (RNE)
// (PR #524 "[Kernel][SM70] Add opt-in E4M3 grouped attention with FP32
// partials", final status: FP32 state until one final combine.)  Weights
// go to shared memory; the O partials are summed by 16 groups of 16 lanes,
// group k taking partitions k, k + 16, ... in ascending order, and the group
// sums in group order: a fixed summation order, so repeated runs agree bit
// for bit.  The row combine kernel runs one group per CTA on barrier 0; the
// barrier id is a parameter so that groups could share a CTA.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "params.h"
#include "verify_attn_e4m3.h"

namespace vae4 {

constexpr int kRowThreads = 256;
constexpr int kRowLanes = 16;                         // float4 lanes: 64 d per unit
constexpr int kRowGroups = kRowThreads / kRowLanes;   // partition groups

// shared scratch of one group: weights and sums of up to P partitions, the
// warp reductions, the group sums
struct RowScratch {
  float *wm, *wl;              // [P] each
  float *red;                  // [kRowThreads / 32]
  float4 (*accs)[kRowLanes];   // [kRowGroups][kRowLanes]
};

__device__ __forceinline__ void row_bar(int id) {
  asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(kRowThreads) : "memory");
}
__device__ __forceinline__ bool row_bar_or(int id, bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n"
      " barrier.red.or.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"(v ? 1u : 0u), "r"(id), "r"(kRowThreads)
      : "memory");
  return r != 0;
}

// slot0 / nP: the unit's stream's first partition slot and partition count
// (nP = 0 for a row without a live query: zeros); sv: the head's V scale.
// tid in [0, 256).
__device__ __forceinline__ void combine_row_unit(const CombineParams &p, int b, int h, int r,
                                                 int dsl, int slot0, int nP, float sv, int tid,
                                                 int bar_id, const RowScratch &sc) {
  const int lane = tid & 31, warp = tid >> 5;
  const int i = r / p.G, g = r - i * p.G;
  const int d0 = dsl * 64;
  __half *out = static_cast<__half *>(p.out) + (int64_t)b * p.o_sb + (int64_t)i * p.o_si +
                (int64_t)(h * p.G + g) * p.o_sh + d0;
  float *wm = sc.wm, *wl = sc.wl;
  const int64_t pstride = (int64_t)p.rows_pad;  // rows per partition
  const float *ml = p.ws_ml + (int64_t)slot0 * pstride * 2 + r * 2;
  const float kNegInf = -__int_as_float(0x7f800000);

  // the first kPre P.V partials of this thread's group are requested now,
  // together with the (m, l) pairs, so both L2 round trips overlap
  const int l4 = tid % kRowLanes, grp = tid / kRowLanes;
  const float *o = p.ws_o + (int64_t)slot0 * pstride * p.D + (int64_t)r * p.D + d0 + 4 * l4;
  const int64_t ostride = pstride * p.D;
  constexpr int kPre = 10;  // covers 160 partitions
  float4 pre[kPre];
#pragma unroll
  for (int k = 0; k < kPre; ++k) {
    const int q = grp + k * kRowGroups;
    pre[k] = q < nP ? __ldcg(reinterpret_cast<const float4 *>(o + q * ostride))
                    : make_float4(0.f, 0.f, 0.f, 0.f);
  }

  // ---- pass 1: (m_p, l_p), maximum over partitions with l_p > 0
  float mx = kNegInf;
  bool bad = false;
  for (int q = tid; q < nP; q += kRowThreads) {
    const float2 v = __ldcg(reinterpret_cast<const float2 *>(ml + q * pstride * 2));
    wm[q] = v.x;
    wl[q] = v.y;
    if (v.y < 0.f) bad = true;  // a partition met an invalid page or timed out
    if (v.y > 0.f) mx = fmaxf(mx, v.x);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  if (lane == 0) sc.red[warp] = mx;
  const bool any_bad = row_bar_or(bar_id, bad);
  float M = sc.red[0];
#pragma unroll
  for (int k = 1; k < kRowThreads / 32; ++k) M = fmaxf(M, sc.red[k]);
  row_bar(bar_id);

  // ---- pass 2: weights w_p = 2^(m_p - M) and the total sum (fixed tree)
  float lam = 0.f;
  for (int q = tid; q < nP; q += kRowThreads) {
    const float l = wl[q];
    const float w = l > 0.f ? (wm[q] == M ? 1.f : exp2f(wm[q] - M)) : 0.f;
    wm[q] = w;
    lam += w * l;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) lam += __shfl_xor_sync(0xffffffffu, lam, off);
  if (lane == 0) sc.red[warp] = lam;
  row_bar(bar_id);
  float Lam = 0.f;
#pragma unroll
  for (int k = 0; k < kRowThreads / 32; ++k) Lam += sc.red[k];

  // ---- pass 3: sum of w_p * O_p over this slice, per group (ascending p),
  // then over groups
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int k = 0; k < kPre; ++k) {
    const int q = grp + k * kRowGroups;
    if (q < nP) {
      const float w = wm[q];
      acc.x += w * pre[k].x;
      acc.y += w * pre[k].y;
      acc.z += w * pre[k].z;
      acc.w += w * pre[k].w;
    }
  }
#pragma unroll 4
  for (int q = grp + kPre * kRowGroups; q < nP; q += kRowGroups) {
    const float w = wm[q];
    const float4 v = __ldcg(reinterpret_cast<const float4 *>(o + q * ostride));
    acc.x += w * v.x;
    acc.y += w * v.y;
    acc.z += w * v.z;
    acc.w += w * v.w;
  }
  sc.accs[grp][l4] = acc;
  row_bar(bar_id);
  if (grp == 0) {
    float4 s = sc.accs[0][l4];
#pragma unroll
    for (int k = 1; k < kRowGroups; ++k) {
      const float4 v = sc.accs[k][l4];
      s.x += v.x;
      s.y += v.y;
      s.z += v.z;
      s.w += v.w;
    }
    uint2 res = make_uint2(0u, 0u);
    if (nP > 0 && !any_bad && Lam > 0.f) {
      const float beta = sv * 256.0f;  // partials hold dec(V) * 2^-8
      const __half2 lo = __floats2half2_rn(__fdiv_rn(s.x, Lam) * beta, __fdiv_rn(s.y, Lam) * beta);
      const __half2 hi = __floats2half2_rn(__fdiv_rn(s.z, Lam) * beta, __fdiv_rn(s.w, Lam) * beta);
      res.x = *reinterpret_cast<const uint32_t *>(&lo);
      res.y = *reinterpret_cast<const uint32_t *>(&hi);
    }
    *reinterpret_cast<uint2 *>(out + 4 * l4) = res;
  }
  row_bar(bar_id);  // the scratch is reused by the group's next unit
}

}  // namespace vae4
