// Device-side balanced partition plan (graph-safe: computed from the lengths
// on the device at every launch).  Every stream (sequence b, KV head h) with
// L live tokens is cut into P_b = ceil(L / W) partitions of W tokens, W the
// same for all streams: a multiple of 16 (at least 64) with
// sum_b Hkv * P_b <= G, the grid's CTA count, so the whole batch runs in one
// wave of equal-sized partitions whatever the mix of lengths.  W starts at
// ceil(sum L / (G / Hkv)) rounded up to 16 and, if that does not fit, is
// bisected (at most six steps) towards a bound that always fits.  At equal
// lengths it is the static plan.  Partitions are numbered b-major, then h,
// then p; partition x is CTA x and workspace slot x.  One warp evaluates
// the plan (lanes over sequences, B <= 1024).
//
// The arithmetic is written once, over a source of live lengths: the split
// kernel stages them in shared memory, the combine reads global memory; the
// same lengths give every kernel the same plan.
#pragma once

#include <stdint.h>

namespace vae4 {

struct PlanIn {
  const int32_t *seq;  // i32 [B] or [B][2] (L, q_len)
  int32_t seq_sb, has_qlen, Qmax, capacity, B, Hkv, G;
};

// Live tokens of sequence b: 0 for invalid or empty sequences (they get no
// partition; the combine reports their status and writes zeros).
__device__ __forceinline__ int live_len(int L, int ql, int Qmax, int capacity) {
  return (L <= 0 || L > capacity || ql <= 0 || ql > Qmax || ql > L) ? 0 : L;
}
__device__ __forceinline__ int plan_live_len(const PlanIn &in, int b) {
  const int L = in.seq[(int64_t)b * in.seq_sb];
  const int ql = in.has_qlen ? in.seq[(int64_t)b * in.seq_sb + 1] : in.Qmax;
  return live_len(L, ql, in.Qmax, in.capacity);
}

// Static grid with P partitions per sequence and T taken from the length
// (the automatic plan of a single sequence): ceil(L / P) rounded up to a
// multiple of 16 (callers raise it to at least 64), so ceil(L / T) <= P.
__device__ __forceinline__ int plan_t_from_len(int L, int P) {
  return (int)(((unsigned)L + (unsigned)P - 1u) / (unsigned)P + 15u) & ~15;
}

// Length sources: len(b) for the b = lane + 32k a loop visits.
struct LenGlobal {  // straight from the lengths array
  PlanIn in;
  __device__ __forceinline__ int operator()(int b) const { return plan_live_len(in, b); }
};
struct LenReg {  // B <= 32: lane b holds L_b (loops visit b = lane only)
  int v;
  __device__ __forceinline__ int operator()(int) const { return v; }
};
struct LenStaged {  // (L, q_len) pairs staged in shared memory
  const int *Ls;
  int Qmax, capacity;
  __device__ __forceinline__ int operator()(int b) const {
    return live_len(Ls[2 * b], Ls[2 * b + 1], Qmax, capacity);
  }
};

__device__ __forceinline__ int warp_sum_i(int v) { return (int)__reduce_add_sync(0xffffffffu, (unsigned)v); }

// sum_b ceil(L_b / W) over the batch (whole warp, result in every lane).
// At every W plan_width tries, the count is at most sum / W + live <= 2G.
template <class Len>
__device__ __forceinline__ int plan_count(const Len &len, int B, int W, int lane) {
  int c = 0;
  for (int b = lane; b < B; b += 32) c += (len(b) + W - 1) / W;
  return warp_sum_i(c);
}

// ceil((H * 2^16 + Lo) / d) for H < 2^26, Lo < 2^32, 0 < d < 2^16, the
// quotient below 2^31: two 32-bit divisions instead of a 64-bit one.
__device__ __forceinline__ int ceil_div_split(unsigned H, unsigned Lo, unsigned d) {
  H += Lo >> 16;
  Lo &= 0xFFFFu;
  const unsigned q1 = H / d, r1 = H - q1 * d;   // r1 < 2^16
  const unsigned t = (r1 << 16) | Lo;           // < 2^32
  const unsigned q2 = t / d, r2 = t - q2 * d;
  return (int)((q1 << 16) + q2 + (r2 != 0));
}

// The partition length W (whole warp; every lane returns the same value).
// B <= 1024: a lane's share of the token sum is below 2^36, so its two
// 16-bit halves reduce without overflow; G / Hkv < 2^16.
template <class Len>
__device__ __forceinline__ int plan_width(const Len &len, int B, int Hkv, int G, int lane) {
  unsigned long long s = 0;
  unsigned nl = 0, mx = 0;
  for (int b = lane; b < B; b += 32) {
    const int L = len(b);
    s += (unsigned)L;
    nl += L > 0;
    mx = max(mx, (unsigned)L);
  }
  const unsigned sH = __reduce_add_sync(0xffffffffu, (unsigned)(s >> 16));
  const unsigned sL = __reduce_add_sync(0xffffffffu, (unsigned)(s & 0xFFFFu));
  const int nlive = (int)__reduce_add_sync(0xffffffffu, nl);
  const int maxL = (int)__reduce_max_sync(0xffffffffu, mx);
  if (nlive == 0) return 64;
  const int gb = G / Hkv;  // partitions per KV head the grid holds (>= nlive)
  auto up16 = [](int x) { return (x + 15) & ~15; };
  // every term is at most maxL < 2^31, so are the quotients (nlive <= gb)
  int lo = max(64, up16(ceil_div_split(sH, sL, (unsigned)gb)));
  if (plan_count(len, B, lo, lane) <= gb) return lo;
  // W that always fits: sum / W + nlive <= gb, or one partition per sequence
  int hi = gb > nlive ? max(lo, up16(ceil_div_split(sH, sL, (unsigned)(gb - nlive))))
                      : max(64, up16(maxL));
  for (int it = 0; it < 6 && hi - lo > 16; ++it) {  // lo fails, hi fits
    const int mid = (int)(((long long)lo + hi) / 32 * 16);
    if (plan_count(len, B, mid, lane) <= gb)
      hi = mid;
    else
      lo = mid;
  }
  return hi;
}

// Partition x -> (b, h, p) and the sequence's partition count; false if x
// is past the last partition.  Whole warp.
template <class Len>
__device__ __forceinline__ bool plan_locate(const Len &len, int B, int Hkv, int W, int x, int lane,
                                            int *b_out, int *h_out, int *p_out, int *np_out) {
  int base = 0;
  for (int b0 = 0; b0 < B; b0 += 32) {
    const int b = b0 + lane;
    const int np = b < B ? (len(b) + W - 1) / W : 0;
    const int cnt = np * Hkv;
    int incl = cnt;  // inclusive scan over the lanes
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    const int excl = incl - cnt;
    const unsigned hit = __ballot_sync(0xffffffffu, cnt > 0 && x >= base + excl && x < base + incl);
    if (hit) {
      const int src = __ffs(hit) - 1;
      const int e = __shfl_sync(0xffffffffu, excl, src);
      const int n = __shfl_sync(0xffffffffu, np, src);
      const int r = x - base - e;
      const int hh = Hkv == 1 ? 0 : r / n;
      *b_out = b0 + src;
      *h_out = hh;
      *p_out = r - hh * n;
      *np_out = n;
      return true;
    }
    base += __shfl_sync(0xffffffffu, incl, 31);
  }
  return false;
}

// Out-of-line entry points (whole warp).  Each kernel evaluates its plan
// once; keeping the code out of the kernel body leaves the body's code
// layout and register allocation as they are without the plan.

// Stage the (L, q_len) pair of every sequence in Ls[2b], Ls[2b + 1]; all of
// a lane's reads of a batch are in flight before the first is stored.
static __device__ __noinline__ void plan_stage(const PlanIn in, int *Ls, int lane) {
  constexpr int kBatch = 8;
  for (int b0 = 0; b0 < in.B; b0 += 32 * kBatch) {
    int vl[kBatch], vq[kBatch];
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const int b = b0 + 32 * k + lane;
      vl[k] = b < in.B ? in.seq[(int64_t)b * in.seq_sb] : 0;
      vq[k] = b < in.B ? (in.has_qlen ? in.seq[(int64_t)b * in.seq_sb + 1] : in.Qmax) : 0;
    }
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const int b = b0 + 32 * k + lane;
      if (b < in.B) {
        Ls[2 * b] = vl[k];
        Ls[2 * b + 1] = vq[k];
      }
    }
  }
  __syncwarp();
}

// CTA x of a split launch, from the staged pairs -> (b, h, p, W); p = -1
// past the end of the plan.
static __device__ __noinline__ int4 plan_cta(const PlanIn in, const int *Ls, int x, int lane) {
  int W, b = -1, h = -1, part = -1, np = 0;
  bool ok;
  if (in.B <= 32) {  // one sequence per lane, in a register
    const LenReg len{lane < in.B ? live_len(Ls[2 * lane], Ls[2 * lane + 1], in.Qmax, in.capacity) : 0};
    W = plan_width(len, in.B, in.Hkv, in.G, lane);
    ok = plan_locate(len, in.B, in.Hkv, W, x, lane, &b, &h, &part, &np);
  } else {
    const LenStaged len{Ls, in.Qmax, in.capacity};
    W = plan_width(len, in.B, in.Hkv, in.G, lane);
    ok = plan_locate(len, in.B, in.Hkv, W, x, lane, &b, &h, &part, &np);
  }
  if (!ok) b = h = part = -1;
  return make_int4(b, h, part, W);
}

// Same, with lengths read from global memory on every pass.
static __device__ __noinline__ int4 plan_cta_global(const PlanIn in, int x, int lane) {
  const LenGlobal len{in};
  const int W = plan_width(len, in.B, in.Hkv, in.G, lane);
  int b = -1, h = -1, part = -1, np = 0;
  if (!plan_locate(len, in.B, in.Hkv, W, x, lane, &b, &h, &part, &np)) b = h = part = -1;
  return make_int4(b, h, part, W);
}

// Stream (b, h) -> (first slot, partition count), from the staged pairs;
// the count is -1 if the stream's slots would run past the grid (never: the
// plan fits by construction).
static __device__ __noinline__ int2 plan_stream_slots(const PlanIn in, const int *Ls, int b, int h,
                                                      int lane) {
  const LenStaged len{Ls, in.Qmax, in.capacity};
  const int W = plan_width(len, in.B, in.Hkv, in.G, lane);
  int before = 0;
  for (int b1 = lane; b1 < b; b1 += 32) before += (len(b1) + W - 1) / W;
  before = warp_sum_i(before);
  int np = (len(b) + W - 1) / W;
  const int s0 = before * in.Hkv + h * np;
  if (s0 + np > in.G) np = -1;
  return make_int2(s0, np);
}

}  // namespace vae4
