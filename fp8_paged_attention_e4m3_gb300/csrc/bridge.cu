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
// bits, s 24, so the FP32 product may be inexact): the product is rounded
// to FP32 to odd and then to FP16 to nearest even (see mul_round_to_odd);
// scales too large for that path's pre-shift take mul_round_fp16 instead,
// which breaks an FP16 tie at the FP32 product by the sign of its exact FMA
// residual.  With the raw flag: dec(byte) itself (exact).
//
// One warp per (b, h, logical page) at a time: the page's K and V slices
// are read in passes of 256 bytes (8 per lane, coalesced), eight passes per
// round with every load in flight before the first conversion, and each
// lane writes its 8 values as one 16-byte store (512 contiguous bytes per
// warp instruction, streaming).
#include <type_traits>

#include "common.cuh"
#include "kernels.h"
#include "verify_attn_e4m3.h"

namespace vae4 {

namespace {

constexpr int kBridgeThreads = 256;
constexpr int kRound = 8;  // 256-byte passes per round

// fp16 of the exact product d * s (d exact in FP32), round to nearest even
__device__ __forceinline__ __half mul_round_fp16(float d, float s) {
  const float p = d * s;
  const float e = fmaf(d, s, -p);  // p + e == d * s exactly
  const __half rn = __float2half_rn(p);
  // p can only be an FP16 tie (the one case where rounding p differs from
  // rounding p + e) if its 12 low fraction bits are zero
  if (e == 0.f || (__float_as_uint(p) & 0xFFFu) != 0u) return rn;
  const __half lo = __float2half_rd(p), hi = __float2half_ru(p);
  if (__half_as_ushort(lo) == __half_as_ushort(hi)) return rn;  // p is an FP16 value
  const float mid = 0.5f * (__half2float(lo) + __half2float(hi));  // exact
  if (p != mid) return rn;
  return e > 0.f ? hi : lo;
}

// FP8 byte b -> dec(b) * 2^-K exactly as an FP32 bit move: the magnitude
// bits land in FP32 bits 26..20 (E4M3, K = 120) or 27..21 (E5M2, K = 112),
// so the FP8 exponent field becomes the low bits of the FP32 one and FP8
// subnormals become FP32 subnormals with the same significand.  (The
// infinity and NaN codes, outside the contract, give finite values.)
template <bool E5M2>
__device__ __forceinline__ float fp8_to_f32_shifted(uint32_t b) {
  return __uint_as_float(((b & 0x80u) << 24) | ((b & 0x7Fu) << (E5M2 ? 21 : 20)));
}
template <bool E5M2>
constexpr float fp8_shift_scale() {  // 2^K
  return E5M2 ? 5.192296858534828e+33f : 1.329227995784916e+36f;
}

// Scaled path: d' = dec(b) 2^-K and s' = s 2^K give the same exact product
// d s.  It is rounded to FP32 *to odd* (toward zero, then the last bit set
// if anything was cut off, which the FMA residual tells), and that value to
// FP16 to nearest even: since FP32 carries at least two more bits than FP16
// (also for FP16 subnormal results), the two roundings give exactly the
// single rounding of d s (Boldo and Melquiond, "When double rounding is
// odd", 2005; "Emulation of FMA and correctly rounded sums: proved
// algorithms using rounding to odd", IEEE Trans. Computers 2008).  Two
// products go to FP16 in one conversion; no branch.
__device__ __forceinline__ float mul_round_to_odd(float d, float s) {
  const float r = __fmul_rz(d, s);
  const float e = __fmaf_rn(d, s, -r);  // d s - r, exact
  return __uint_as_float(__float_as_uint(r) | (e != 0.f ? 1u : 0u));
}
template <bool E5M2>
__device__ __forceinline__ uint32_t scaled_pair(uint32_t b0, uint32_t b1, float s2) {
  const float p0 = mul_round_to_odd(fp8_to_f32_shifted<E5M2>(b0), s2);
  const float p1 = mul_round_to_odd(fp8_to_f32_shifted<E5M2>(b1), s2);
  const __half2 h = __floats2half2_rn(p0, p1);
  return *reinterpret_cast<const uint32_t *>(&h);
}

// 8 FP8 bytes -> 8 FP16 values (scaled unless RAW); with SHIFT, sc is s * 2^K
template <bool E5M2, bool RAW, bool SHIFT>
__device__ __forceinline__ uint4 convert8(uint2 raw, float sc) {
  if constexpr (!RAW && SHIFT) {
    const uint32_t x = raw.x, y = raw.y;
    return make_uint4(scaled_pair<E5M2>(x & 0xFFu, (x >> 8) & 0xFFu, sc),
                      scaled_pair<E5M2>((x >> 16) & 0xFFu, x >> 24, sc),
                      scaled_pair<E5M2>(y & 0xFFu, (y >> 8) & 0xFFu, sc),
                      scaled_pair<E5M2>((y >> 16) & 0xFFu, y >> 24, sc));
  }
  const uint32_t wds[2] = {raw.x, raw.y};
  uint32_t hw[4];
#pragma unroll
  for (int e = 0; e < 2; ++e) {
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
  return make_uint4(hw[0], hw[1], hw[2], hw[3]);
}

template <bool E5M2, bool RAW>
__global__ void __launch_bounds__(kBridgeThreads) bridge_kernel(const BridgeParams p) {
  const int warps = gridDim.x * (kBridgeThreads / 32);
  const int w = blockIdx.x * (kBridgeThreads / 32) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
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
      float sk = RAW ? 1.f : p.scales[h * p.scale_sh + 0];
      float sv = RAW ? 1.f : p.scales[h * p.scale_sh + 1];
      // pre-shifted scales for the bit-move decode, exact while finite
      // (scales below 2^(127 - K)); otherwise the general path
      const float sk2 = sk * fp8_shift_scale<E5M2>(), sv2 = sv * fp8_shift_scale<E5M2>();
      const bool shift = !RAW && isfinite(sk2) && isfinite(sv2) && sk2 != 0.f && sv2 != 0.f;
      if (shift) {
        sk = sk2;
        sv = sv2;
      }
      const int64_t slice = (int64_t)p.page * p.D;
      const uint8_t *k = p.kv + ((int64_t)(ok_page ? phys : 0) * 2 * p.Hkv + h) * slice;
      const uint8_t *v = k + (int64_t)p.Hkv * slice;
      uint16_t *ko = p.k_out + (int64_t)b * p.o_sb + (int64_t)h * p.o_sh +
                     (int64_t)lp * p.page * p.o_st;
      uint16_t *vo = p.v_out + (int64_t)b * p.o_sb + (int64_t)h * p.o_sh +
                     (int64_t)lp * p.page * p.o_st;
      const int nbytes = toks * p.D;  // bytes of this page's slice that are live
      // one copy of the loop per conversion path (the choice is per page)
      auto rounds = [&](auto shift_tag) {
        constexpr bool SH = decltype(shift_tag)::value;
        for (int base = 0; base < nbytes; base += kRound * 256) {
          uint2 rk[kRound], rv[kRound];
#pragma unroll
          for (int j = 0; j < kRound; ++j) {
            const int off = base + 256 * j + 8 * lane;
            rk[j] = rv[j] = make_uint2(0u, 0u);
            if (ok_page && off < nbytes) {
              rk[j] = __ldcs(reinterpret_cast<const uint2 *>(k + off));
              rv[j] = __ldcs(reinterpret_cast<const uint2 *>(v + off));
            }
          }
#pragma unroll
          for (int j = 0; j < kRound; ++j) {
            const int off = base + 256 * j + 8 * lane;
            if (off < nbytes) {
              const int t = off / p.D, d = off - t * p.D;
              const int64_t o = (int64_t)t * p.o_st + d;
              __stcs(reinterpret_cast<uint4 *>(ko + o), convert8<E5M2, RAW, SH>(rk[j], sk));
              __stcs(reinterpret_cast<uint4 *>(vo + o), convert8<E5M2, RAW, SH>(rv[j], sv));
            }
          }
        }
      };
      if (shift)
        rounds(std::true_type{});
      else
        rounds(std::false_type{});
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
