// Combine kernel: merges the FP32 partition states of each output row in
// ascending partition order and writes the FP16 output.
//
// For row r of (sequence b, KV head h), over the live partitions p (those
// with p*T < L and a nonzero running sum):
//     M   = max_p m_p                  (m_p in log2 units of the score)
//     w_p = 2^(m_p - M)
//     out = (sum_p w_p O_p) / (sum_p w_p l_p) * s_V * 2^8
// all in FP32, rounded once to FP16 (round to nearest even), with a fixed
// summation order.  It is the one place where the FP32 partition state
// (max, sum, unnormalised P.V) is reduced, and it reduces in FP32 (PR #524
// "[Kernel][SM70] Add opt-in E4M3 grouped attention with FP32 partials",
// final status; PR #560 "[Bugfix] Use FP32 state and E4M3 defaults for
// DFlash2", Purpose).
// Padding query slots, dead sequences (L == 0) and sequences whose lengths
// or pages were invalid get zeros.
#include "common.cuh"
#include "kernels.h"
#include "plan.cuh"
#include "verify_attn_e4m3.h"

namespace vae4 {

namespace {

constexpr int kCombineThreads = 256;
constexpr int kLanes = 16;                          // float4 lanes: 64 d per CTA
constexpr int kGroups = kCombineThreads / kLanes;   // partition groups

// One CTA per (output row, 64-wide slice of d).  Every CTA of a row computes
// the row's partition weights into shared memory (a few hundred floats);
// the P.V partials of its slice are then summed by kGroups groups of
// threads, group k taking partitions k, k + kGroups, ... in ascending order,
// and the group sums are added in group order: a fixed summation order that
// does not depend on scheduling, so repeated runs agree bit for bit.  Many
// short independent loads per thread keep the L2 busy instead of waiting on
// one long dependent chain.
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(const CombineParams p) {
  extern __shared__ __align__(16) float csm[];
  __shared__ float red[kCombineThreads / 32];
  __shared__ float4 accs[kGroups][kLanes];

  const int nd = p.D / 64;  // d slices per row
  const int r = blockIdx.x / nd, dsl = blockIdx.x - r * nd;
  const int h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int i = r / p.G, g = r - i * p.G;
  const int d0 = dsl * 64;
  __half *out = static_cast<__half *>(p.out) + (int64_t)b * p.o_sb + (int64_t)i * p.o_si +
                (int64_t)(h * p.G + g) * p.o_sh + d0;

  // lengths are inputs of the step, not results of the split kernel: read
  // them before waiting for it
  const int L = p.seq[(int64_t)b * p.seq_sb];
  const int ql = p.seq_has_qlen ? p.seq[(int64_t)b * p.seq_sb + 1] : p.Qmax;
  // partitions of this (sequence, KV head): slots slot0 .. slot0 + nP - 1
  int nP = 0, slot0 = 0;
  if (!p.dev_plan) {
    slot0 = (b * p.Hkv + h) * p.P;
    const int T = (p.t_from_len && L > 0 && L <= p.capacity) ? max(64, plan_t_from_len(L, p.P)) : p.T;
    nP = (L + T - 1) / T;
  }

  // wait until the split kernel's partials are complete and visible
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  bool dead = L <= 0 || L > p.capacity || ql < 0 || ql > p.Qmax || ql > L || i >= ql;
  if (blockIdx.x == 0 && h == 0 && tid == 0) {  // report invalid lengths once per sequence
    if (L < 0 || L > p.capacity) atomicOr(p.status, VAE4_STATUS_BAD_LENGTH);
    else if (ql < 0 || ql > p.Qmax || (L > 0 && ql > L)) atomicOr(p.status, VAE4_STATUS_BAD_QLEN);
  }
  if (p.dev_plan && !dead) {
    // the device-side plan, as the split kernel's CTA of the stream's first
    // partition recorded it (every live row's stream has one)
    const int2 e = p.plan_tab[b * p.Hkv + h];
    slot0 = e.x;
    nP = e.y;
    if (slot0 < 0 || nP < 1 || nP > p.P || slot0 + nP > p.plan_G) {  // never: a library bug
      if (tid == 0) atomicOr(p.status, VAE4_STATUS_PLAN);
      dead = true;
    }
  }
  if (dead) nP = 0;
  float *wm = csm;       // m_p, then the weight w_p
  float *wl = csm + p.P; // l_p
  const int64_t pstride = (int64_t)p.rows_pad;  // rows per partition
  const float *ml = p.ws_ml + (int64_t)slot0 * pstride * 2 + r * 2;
  const float kNegInf = -__int_as_float(0x7f800000);

  // the first kPre P.V partials of this thread's group are requested now,
  // together with the (m, l) pairs, so both L2 round trips overlap
  const int l4 = tid % kLanes, grp = tid / kLanes;
  const float *o = p.ws_o + (int64_t)slot0 * pstride * p.D + (int64_t)r * p.D + d0 + 4 * l4;
  const int64_t ostride = pstride * p.D;
  constexpr int kPre = 10;  // covers 160 partitions
  float4 pre[kPre];
#pragma unroll
  for (int k = 0; k < kPre; ++k) {
    const int q = grp + k * kGroups;
    pre[k] = q < nP ? __ldcg(reinterpret_cast<const float4 *>(o + q * ostride))
                    : make_float4(0.f, 0.f, 0.f, 0.f);
  }

  // ---- pass 1: (m_p, l_p), maximum over partitions with l_p > 0
  float mx = kNegInf;
  bool bad = false;
  for (int q = tid; q < nP; q += kCombineThreads) {
    const float2 v = *reinterpret_cast<const float2 *>(ml + q * pstride * 2);
    wm[q] = v.x;
    wl[q] = v.y;
    if (v.y < 0.f) bad = true;  // a partition met an invalid page or timed out
    if (v.y > 0.f) mx = fmaxf(mx, v.x);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if (lane == 0) red[warp] = mx;
  const bool any_bad = __syncthreads_or(bad);
  float M = red[0];
#pragma unroll
  for (int k = 1; k < kCombineThreads / 32; ++k) M = fmaxf(M, red[k]);
  __syncthreads();

  // ---- pass 2: weights w_p = 2^(m_p - M) and the total sum (fixed tree)
  float lam = 0.f;
  for (int q = tid; q < nP; q += kCombineThreads) {
    const float l = wl[q];
    const float w = l > 0.f ? (wm[q] == M ? 1.f : exp2f(wm[q] - M)) : 0.f;
    wm[q] = w;
    lam += w * l;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) lam += __shfl_xor_sync(0xffffffffu, lam, o);
  if (lane == 0) red[warp] = lam;
  __syncthreads();
  float Lam = 0.f;
#pragma unroll
  for (int k = 0; k < kCombineThreads / 32; ++k) Lam += red[k];

  // ---- pass 3: sum of w_p * O_p over this slice, per group (ascending p),
  // then over groups
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int k = 0; k < kPre; ++k) {
    const int q = grp + k * kGroups;
    if (q < nP) {
      const float w = wm[q];
      acc.x += w * pre[k].x;
      acc.y += w * pre[k].y;
      acc.z += w * pre[k].z;
      acc.w += w * pre[k].w;
    }
  }
#pragma unroll 4
  for (int q = grp + kPre * kGroups; q < nP; q += kGroups) {
    const float w = wm[q];
    const float4 v = __ldcg(reinterpret_cast<const float4 *>(o + q * ostride));
    acc.x += w * v.x;
    acc.y += w * v.y;
    acc.z += w * v.z;
    acc.w += w * v.w;
  }
  accs[grp][l4] = acc;
  __syncthreads();
  if (grp != 0) return;
  float4 s = accs[0][l4];
#pragma unroll
  for (int k = 1; k < kGroups; ++k) {
    const float4 v = accs[k][l4];
    s.x += v.x;
    s.y += v.y;
    s.z += v.z;
    s.w += v.w;
  }
  uint2 res = make_uint2(0u, 0u);
  if (!dead && !any_bad && Lam > 0.f) {
    const float beta = p.scales[h * p.scale_sh + 1] * 256.0f;  // partials hold dec(V) * 2^-8
    const __half2 lo = __floats2half2_rn(__fdiv_rn(s.x, Lam) * beta, __fdiv_rn(s.y, Lam) * beta);
    const __half2 hi = __floats2half2_rn(__fdiv_rn(s.z, Lam) * beta, __fdiv_rn(s.w, Lam) * beta);
    res.x = *reinterpret_cast<const uint32_t *>(&lo);
    res.y = *reinterpret_cast<const uint32_t *>(&hi);
  }
  *reinterpret_cast<uint2 *>(out + 4 * l4) = res;
}

__global__ void decode_table_kernel(uint16_t *out, bool integer_path, bool e5m2) {
  const int t = threadIdx.x;  // 64 threads x 4 codes
  const uint32_t w = (uint32_t)(4 * t) | (uint32_t)(4 * t + 1) << 8 | (uint32_t)(4 * t + 2) << 16 |
                     (uint32_t)(4 * t + 3) << 24;
  uint32_t lo, hi;
  if (e5m2) {
    lo = fp8x2_to_f16x2<true>(w);
    hi = fp8x2_to_f16x2<true>(w >> 16);
  } else if (integer_path) {
    e4m3x4_to_f16x4(w, lo, hi);
  } else {
    e4m3x4_to_f16x4_hw(w, lo, hi);
  }
  out[4 * t + 0] = (uint16_t)(lo & 0xFFFFu);
  out[4 * t + 1] = (uint16_t)(lo >> 16);
  out[4 * t + 2] = (uint16_t)(hi & 0xFFFFu);
  out[4 * t + 3] = (uint16_t)(hi >> 16);
}

}  // namespace

cudaError_t launch_combine(const CombineParams &p, cudaStream_t stream) {
  if (p.D % 64 != 0) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.Qmax * p.G * (p.D / 64), p.Hkv, p.B);
  cfg.blockDim = dim3(kCombineThreads);
  cfg.dynamicSmemBytes = (size_t)p.P * 2 * sizeof(float);  // (m_p, l_p) per partition
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const int smem = (int)cfg.dynamicSmemBytes;
  if (smem > 48 * 1024) {  // beyond the default dynamic shared-memory limit
    const cudaError_t e =
        cudaFuncSetAttribute(combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
  }
  return cudaLaunchKernelEx(&cfg, combine_kernel, p);
}

cudaError_t launch_decode_table(uint16_t *out, bool integer_path, bool e5m2,
                                cudaStream_t stream) {
  decode_table_kernel<<<1, 64, 0, stream>>>(out, integer_path, e5m2);
  return cudaGetLastError();
}

}  // namespace vae4
