// Paged FP8 -> FP16 bridge: writes, for every (sequence b, KV head h), the
// FP16 K and V of tokens 0 .. L-1 into dense [B][Hkv][cap][D] buffers (the
// layout a dense FP16 attention reads), gathering the pages through the
// block table.  The pages describe this call as an explicit E4M3
// paged-to-FP16 bridge next to the grouped attention (PR #524 "[Kernel]
// [SM70] Add opt-in E4M3 grouped attention with FP32 partials", historical
// R6 purpose and scope).
//
// Value written: fp16(dec(byte) * s) with s the head's FP32 K or V scale,
// rounded once from the exact product (dec(byte) has at most 4 significant
// bits, s 24: the FP32 product p may be inexact, but its error e is exact
// from an FMA; an FP16 tie at p -- the only case where rounding p differs
// from rounding p + e, since FP16 midpoints are FP32 numbers -- is broken
// by the sign of e).  With the raw flag: dec(byte) itself (exact).
//
// One warp per (b, h, logical page): each lane converts 16 bytes (16
// elements of one token) per step and stores 32 bytes; K and V interleaved.
#include "common.cuh"
#include "kernels.h"
#include "verify_attn_e4m3.h"

namespace vae4 {

namespace {

constexpr int kBridgeThreads = 256;

// fp16 of the exact product d * s (d exact in FP32), round to nearest even
__device__ __forceinline__ __half mul_round_fp16(float d, float s) {
  const float p = d * s;
  const float e = fmaf(d, s, -p);  // p + e == d * s exactly
  const __half rn = __float2half_rn(p);
  if (e == 0.f) return rn;
  const __half lo = __float2half_rd(p), hi = __float2half_ru(p);
  if (__half_as_ushort(lo) == __half_as_ushort(hi)) return rn;  // p is an FP16 value
  const float mid = 0.5f * (__half2float(lo) + __half2float(hi));  // exact
  if (p != mid) return rn;
  return e > 0.f ? hi : lo;
}

template <bool E5M2, bool RAW>
__global__ void __launch_bounds__(kBridgeThreads) bridge_kernel(const BridgeParams p) {
  const int warps = gridDim.x * (kBridgeThreads / 32);
  const int w = blockIdx.x * (kBridgeThreads / 32) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  const int cpt = p.D / 16;  // 16-byte chunks per token
  for (int b = 0; b < p.B; ++b) {
    const int L = p.seq[(int64_t)b * p.seq_sb];
    if (L < 0 || L > p.cap) {
      if (w == 0 && lane == 0 && p.status) atomicOr(p.status, VAE4_STATUS_BAD_LENGTH);
      continue;
    }
    const int npg = (L + p.page - 1) / p.page;
    const int units = npg * p.Hkv;
    for (int u = w; u < units; u += warps) {
      const int lp = u / p.Hkv, h = u - lp * p.Hkv;
      const int phys = p.bt[(int64_t)b * p.bt_sb + lp];
      const bool ok_page = phys >= 0 && phys < p.n_pages;
      if (!ok_page && lane == 0 && p.status) atomicOr(p.status, VAE4_STATUS_BAD_BLOCK);
      const int toks = min(p.page, L - lp * p.page);
      const float sk = RAW ? 1.f : p.scales[h * p.scale_sh + 0];
      const float sv = RAW ? 1.f : p.scales[h * p.scale_sh + 1];
      const int64_t slice = (int64_t)p.page * p.D;
      const uint8_t *k = p.kv + ((int64_t)(ok_page ? phys : 0) * 2 * p.Hkv + h) * slice;
      const uint8_t *v = k + (int64_t)p.Hkv * slice;
      uint16_t *ko = p.k_out + (int64_t)b * p.o_sb + (int64_t)h * p.o_sh;
      uint16_t *vo = p.v_out + (int64_t)b * p.o_sb + (int64_t)h * p.o_sh;
      const int nch = toks * cpt;
      for (int c = lane; c < nch; c += 32) {
        const int t = c / cpt, d0 = (c - t * cpt) * 16;
        const int64_t orow = (int64_t)(lp * p.page + t) * p.o_st + d0;
        uint4 rk = make_uint4(0, 0, 0, 0), rv = make_uint4(0, 0, 0, 0);
        if (ok_page) {
          rk = __ldcs(reinterpret_cast<const uint4 *>(k + (int64_t)c * 16));
          rv = __ldcs(reinterpret_cast<const uint4 *>(v + (int64_t)c * 16));
        }
#pragma unroll
        for (int kv = 0; kv < 2; ++kv) {
          const uint4 raw = kv ? rv : rk;
          const float sc = kv ? sv : sk;
          const uint32_t wds[4] = {raw.x, raw.y, raw.z, raw.w};
          uint32_t hw[8];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const uint32_t h0 = fp8x2_to_f16x2<E5M2>(wds[e]);
            const uint32_t h1 = fp8x2_to_f16x2<E5M2>(wds[e] >> 16);
            if (RAW) {
              hw[2 * e] = h0;
              hw[2 * e + 1] = h1;
            } else {
              const __half2 a = *reinterpret_cast<const __half2 *>(&h0);
              const __half2 c2 = *reinterpret_cast<const __half2 *>(&h1);
              const __half2 ra = __halves2half2(mul_round_fp16(__low2float(a), sc),
                                                mul_round_fp16(__high2float(a), sc));
              const __half2 rc = __halves2half2(mul_round_fp16(__low2float(c2), sc),
                                                mul_round_fp16(__high2float(c2), sc));
              hw[2 * e] = *reinterpret_cast<const uint32_t *>(&ra);
              hw[2 * e + 1] = *reinterpret_cast<const uint32_t *>(&rc);
            }
          }
          uint4 *dst = reinterpret_cast<uint4 *>((kv ? vo : ko) + orow);
          __stcs(dst, make_uint4(hw[0], hw[1], hw[2], hw[3]));
          __stcs(dst + 1, make_uint4(hw[4], hw[5], hw[6], hw[7]));
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_bridge(const BridgeParams &p, int num_sms, bool e5m2, bool raw,
                          cudaStream_t stream) {
  const int grid = 8 * (num_sms > 0 ? num_sms : 1);
  if (e5m2) {
    if (raw) bridge_kernel<true, true><<<grid, kBridgeThreads, 0, stream>>>(p);
    else bridge_kernel<true, false><<<grid, kBridgeThreads, 0, stream>>>(p);
  } else {
    if (raw) bridge_kernel<false, true><<<grid, kBridgeThreads, 0, stream>>>(p);
    else bridge_kernel<false, false><<<grid, kBridgeThreads, 0, stream>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace vae4
