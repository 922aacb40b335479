// Device-side balanced partition plan (graph-safe: computed from the lengths
// on the device at every launch).  Every stream (sequence b, KV head h) with
// L live tokens is cut into P_b = ceil(L / W) partitions of W tokens, W the
// same for all streams, and each partition runs as r_b CTAs, one per row
// group of N rows that holds a live query (r_b = ceil(q_len * GQA / N)).
// W is a multiple of 16 (at least 64) with sum_b Hkv * r_b * P_b <= G, the
// grid's CTA count, so the whole batch runs in one wave of equal-sized CTAs
// whatever the mix of lengths and query counts.  W starts at
// ceil(sum r L / (G / Hkv)) rounded up to 16 and, if that does not fit, is
// bisected (at most six steps) towards a bound that always fits.  At equal
// lengths it is the static plan.  Partitions are numbered by the sequence's
// row groups (most first), then b, h, p; partition x runs as CTAs
// (x, row group) of a G x (row groups) grid, those of row groups without
// live queries leaving at once, and is workspace slot x.  One warp evaluates the plan (lanes over sequences,
// B <= 1024).
//
// The arithmetic is written once, over a source of (live length, row
// groups) pairs: the tcgen05 split kernel stages the lengths in shared
// memory, the mma.sync one reads global memory.  The CTA of each stream's
// first partition records the stream's first slot and partition count in
// the workspace for the combine.
#pragma once

#include <stdint.h>

namespace vae4 {

struct PlanIn {
  const int32_t *seq;  // i32 [B] or [B][2] (L, q_len)
  int32_t seq_sb, has_qlen, Qmax, capacity, B, Hkv, G;
  int32_t gqa, N;      // query heads per KV head; rows per CTA (a row group)
};

// Row groups a sequence with q_len queries keeps busy (0 if not live).
__device__ __forceinline__ int plan_row_groups(int L_live, int ql, int gqa, int N) {
  return L_live > 0 ? (ql * gqa + N - 1) / N : 0;
}

// Live tokens of sequence b: 0 for invalid or empty sequences (they get no
// partition; the combine reports their status and writes zeros).
__device__ __forceinline__ int live_len(int L, int ql, int Qmax, int capacity) {
  return (L <= 0 || L > capacity || ql <= 0 || ql > Qmax || ql > L) ? 0 : L;
}


// Static grid with P partitions per sequence and T taken from the length
// (the automatic plan of a single sequence): ceil(L / P) rounded up to a
// multiple of 16 (callers raise it to at least 64), so ceil(L / T) <= P.
__device__ __forceinline__ int plan_t_from_len(int L, int P) {
  return (int)(((unsigned)L + (unsigned)P - 1u) / (unsigned)P + 15u) & ~15;
}

// Sources of (live length, row groups) per sequence: len(b) for the
// b = lane + 32k a loop visits.
struct LenGlobal {  // straight from the lengths array
  PlanIn in;
  __device__ __forceinline__ int2 operator()(int b) const {
    const int L = in.seq[(int64_t)b * in.seq_sb];
    const int ql = in.has_qlen ? in.seq[(int64_t)b * in.seq_sb + 1] : in.Qmax;
    const int Ll = live_len(L, ql, in.Qmax, in.capacity);
    return make_int2(Ll, plan_row_groups(Ll, ql, in.gqa, in.N));
  }
};
struct LenReg {  // B <= 32: lane b holds its pair (loops visit b = lane only)
  int2 v;
  __device__ __forceinline__ int2 operator()(int) const { return v; }
};
struct LenStaged {  // (L, q_len) pairs staged in shared memory
  const int *Ls;
  int Qmax, capacity, gqa, N;
  __device__ __forceinline__ int2 operator()(int b) const {
    const int ql = Ls[2 * b + 1];
    const int Ll = live_len(Ls[2 * b], ql, Qmax, capacity);
    return make_int2(Ll, plan_row_groups(Ll, ql, gqa, N));
  }
};

__device__ __forceinline__ int warp_sum_i(int v) { return (int)__reduce_add_sync(0xffffffffu, (unsigned)v); }

// sum_b r_b * ceil(L_b / W) over the batch (whole warp, result in every
// lane).  At every W plan_width tries, the count is at most
// sum r L / W + sum r <= 2G.
template <class Len>
__device__ __forceinline__ int plan_count(const Len &len, int B, int W, int lane) {
  int c = 0;
  for (int b = lane; b < B; b += 32) {
    const int2 v = len(b);
    c += v.y * ((v.x + W - 1) / W);
  }
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
// B <= 1024 and r <= 8: a lane's share of the weighted token sum is below
// 2^39, so its two 16-bit halves reduce without overflow; G / Hkv < 2^16.
template <class Len>
__device__ __forceinline__ int plan_width(const Len &len, int B, int Hkv, int G, int lane) {
  unsigned long long s = 0;
  unsigned nr = 0, mx = 0;
  for (int b = lane; b < B; b += 32) {
    const int2 v = len(b);
    s += (unsigned long long)v.x * (unsigned)v.y;
    nr += v.y;
    mx = max(mx, (unsigned)v.x);
  }
  const unsigned sH = __reduce_add_sync(0xffffffffu, (unsigned)(s >> 16));
  const unsigned sL = __reduce_add_sync(0xffffffffu, (unsigned)(s & 0xFFFFu));
  const int nrg = (int)__reduce_add_sync(0xffffffffu, nr);  // live (sequence, row group)s
  const int maxL = (int)__reduce_max_sync(0xffffffffu, mx);
  if (nrg == 0) return 64;
  const int gb = G / Hkv;  // CTAs per KV head the grid holds (>= nrg)
  auto up16 = [](int x) { return (int)min(((long long)x + 15) & ~15ll, 0x7FFFFFF0ll); };
  // every term is at most maxL < 2^31, so is this quotient (nrg <= gb)
  int lo = max(64, up16(ceil_div_split(sH, sL, (unsigned)gb)));
  if (plan_count(len, B, lo, lane) <= gb) return lo;
  // W that always fits: one partition per sequence, or sum r L / W + nrg <= gb
  // (taken when smaller and its quotient is far from overflow)
  int hi = max(64, up16(maxL));
  if (gb > nrg) {
    const unsigned d = (unsigned)(gb - nrg);
    if ((sH + (sL >> 16)) / d < (1u << 14)) hi = min(hi, up16(ceil_div_split(sH, sL, d)));
  }
  hi = max(hi, lo);
  for (int it = 0; it < 6 && hi - lo > 16; ++it) {  // lo fails, hi fits
    const int mid = (int)(((long long)lo + hi) / 32 * 16);
    if (plan_count(len, B, mid, lane) <= gb)
      hi = mid;
    else
      lo = mid;
  }
  return hi;
}

// Where partition x of the plan sits (whole warp).
struct PlanCta {
  int b, h, p;  // sequence, KV head, partition
  int W;        // the plan's partition length
  int np;       // partitions of the stream
};

// Most row groups a sequence can keep busy (Qmax queries).
__device__ __forceinline__ int plan_max_row_groups(const PlanIn &in) {
  return (in.Qmax * in.gqa + in.N - 1) / in.N;
}

// Partition x -> (b, h, p); false if x is past the last partition.
// Partitions are numbered by row groups (most first), then b, h, p: with
// the row group as grid.y, the CTAs that row groups past the first keep
// busy are the lowest x, launched first in their grid row.
template <class Len>
__device__ __forceinline__ bool plan_locate(const Len &len, int B, int Hkv, int W, int rmax, int x,
                                            int lane, PlanCta *out) {
  int base = 0;  // partitions numbered before this chunk
  for (int rc = rmax; rc >= 1; --rc) {
    for (int b0 = 0; b0 < B; b0 += 32) {
      const int b = b0 + lane;
      int2 v = make_int2(0, 0);
      if (b < B) v = len(b);
      const int np = v.y == rc ? (v.x + W - 1) / W : 0;
      const int cnt = np * Hkv;
      int incl = cnt;  // inclusive scan over the lanes
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      const int excl = incl - cnt;
      const unsigned hit = __ballot_sync(0xffffffffu, cnt > 0 && x >= base + excl && x < base + incl);
      if (hit) {
        const int src = __ffs(hit) - 1;
        const int e = __shfl_sync(0xffffffffu, excl, src);
        const int n = __shfl_sync(0xffffffffu, np, src);
        const int r = x - base - e;
        const int hh = Hkv == 1 ? 0 : r / n;
        out->b = b0 + src;
        out->h = hh;
        out->p = r - hh * n;
        out->np = n;
        return true;
      }
      base += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  return false;
}

// Row group of the plan's CTA c, CTAs numbered row group by row group:
// row group k has one CTA per partition of the sequences that keep more
// than k row groups busy, which the partition numbering puts first, so CTA
// c of row group k serves partition *c (returned through c) and the live
// CTAs are exactly the first sum_b Hkv r_b P_b.  -1 past the plan.
template <class Len>
__device__ __forceinline__ int plan_row_group(const Len &len, int B, int Hkv, int W, int rmax,
                                              int *c, int lane) {
  for (int k = 0; k < rmax; ++k) {
    int cnt = 0;
    for (int b = lane; b < B; b += 32) {
      const int2 v = len(b);
      if (v.y > k) cnt += (v.x + W - 1) / W;
    }
    const int np = warp_sum_i(cnt) * Hkv;
    if (*c < np) return k;
    *c -= np;
  }
  return -1;
}

// Out-of-line entry points (whole warp).  Each kernel evaluates its plan
// once; keeping the code out of the kernel body leaves the body's code
// layout and register allocation close to what they are without the plan.

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

// CTA c of a split launch (one CTA per live (partition, row group), row
// groups in turn: plan_row_group), from the staged pairs, with the plan's
// W; p = -1 past the end of the plan.  Lane 0 also stores the CTA's
// partition number (its workspace slot) and row group at xr[0], xr[1]
// (0 and 0 past the plan).
static __device__ __noinline__ PlanCta plan_cta(const PlanIn in, const int *Ls, int cta, int lane,
                                                volatile int *xr) {
  PlanCta c{-1, -1, -1, 0, 0};
  int W, x = cta, rg = -1;
  bool ok;
  if (in.B <= 32) {  // one sequence per lane, in registers
    int2 v = make_int2(0, 0);
    if (lane < in.B) {
      const int ql = Ls[2 * lane + 1];
      const int Ll = live_len(Ls[2 * lane], ql, in.Qmax, in.capacity);
      v = make_int2(Ll, plan_row_groups(Ll, ql, in.gqa, in.N));
    }
    const LenReg len{v};
    W = plan_width(len, in.B, in.Hkv, in.G, lane);
    rg = plan_row_group(len, in.B, in.Hkv, W, plan_max_row_groups(in), &x, lane);
    ok = rg >= 0 && plan_locate(len, in.B, in.Hkv, W, plan_max_row_groups(in), x, lane, &c);
  } else {
    const LenStaged len{Ls, in.Qmax, in.capacity, in.gqa, in.N};
    W = plan_width(len, in.B, in.Hkv, in.G, lane);
    rg = plan_row_group(len, in.B, in.Hkv, W, plan_max_row_groups(in), &x, lane);
    ok = rg >= 0 && plan_locate(len, in.B, in.Hkv, W, plan_max_row_groups(in), x, lane, &c);
  }
  if (!ok) c = PlanCta{-1, -1, -1, 0, 0};
  c.W = W;
  if (lane == 0) {
    xr[0] = ok ? x : 0;
    xr[1] = ok ? rg : 0;
  }
  return c;
}

// Same, with lengths read from global memory on every pass.
static __device__ __noinline__ PlanCta plan_cta_global(const PlanIn in, int x, int lane) {
  PlanCta c{-1, -1, -1, 0, 0};
  const LenGlobal len{in};
  const int W = plan_width(len, in.B, in.Hkv, in.G, lane);
  if (!plan_locate(len, in.B, in.Hkv, W, plan_max_row_groups(in), x, lane, &c))
    c = PlanCta{-1, -1, -1, 0, 0};
  c.W = W;
  return c;
}

}  // namespace vae4
