// Split (partition) kernel on the 5th-generation tensor cores (tcgen05, TMEM
// accumulators, TMA tensor loads) -- the production path on sm_103a.
//
// One CTA = one (partition p, KV head h and row group, sequence b).  The
// context is walked in 128-key tiles made of two 64-key half-tiles.
// Warp roles (20 warps):
//
//   K / V producer  : one warp each walks the block table (32 entries per
//                     load, prefetched one batch ahead into registers, the
//                     first batch before the CTA's set-up) and issues TMA
//                     tensor loads (128-byte swizzle), one 16 x D byte page
//                     slice per load, of the E4M3 K (resp. V) of a half-tile
//                     into its own ring of raw slots (5-8 slots each: the
//                     shared memory holds only raw bytes, Q and P).  Keys
//                     past the partition and pages with invalid ids are
//                     loaded from outside the tensor, which fills zeros.
//   K decoders (4)  : thread = key; exact E4M3 -> FP16 with the hardware
//                     converter, straight into tensor memory: the A operand
//                     of S^T = K . Q^T (lane = key, column = pair of d).
//                     With N = 16 rows the next tile's decode of each 128-d
//                     half starts once this tile's score MMAs of that half
//                     are done.
//   V decoders (4)  : warp = 32 d of every 128-d block, all 64 keys of a
//                     half-tile: a transposing 8-bit ldmatrix of 16 keys x
//                     16 d gives each thread four consecutive keys of one d,
//                     which after the same exact conversion is a 16x256b
//                     tensor-memory store fragment: V^T lands in TMEM as the
//                     A operand of O^T = V^T . P^T (lane = d, column = pair
//                     of keys), in a ring of 2-4 half-tile slots.
//   score MMA warp  : issues tcgen05.mma.kind::f16  S^T[128 x N] = K . Q^T
//   value MMA warp  : issues tcgen05.mma.kind::f16  O^T[d x N] += V^T . P^T
//                     (both with A in TMEM and B in shared memory; FP32
//                     accumulators in TMEM; commits to mbarriers).  One
//                     lane of each issues the whole chain: a warp-uniform
//                     loop with an elected issuer was faster alone but
//                     slower in this kernel.
//   softmax (8)     : thread = key, half of the N rows each; loads S^T from
//                     TMEM, applies the causal / partition mask at the
//                     edges, keeps the FP32 running max per row (raised
//                     lazily: only when a score exceeds it by more than 2^12,
//                     then running sums and TMEM O^T columns are rescaled),
//                     writes P = 2^(t - m) as FP16 and adds the same rounded
//                     P into FP32 per-row sums.
//
// Rows are (query i, group head g) pairs r = i*G + g of KV head h; N of them
// (<= 64) per CTA form the N dimension of both products (48 for q8 GQA6).
// The partition's FP32 (max, sum, unnormalised P.V) go to the workspace for
// the combine kernel, the only place they are merged (PR #524 "[Kernel][SM70]
// Add opt-in E4M3 grouped attention with FP32 partials", final status).  Keys are visited in ascending logical
// order, so the result does not depend on where pages live.
//
// Every mbarrier wait is bounded; on expiry the CTA raises an abort flag,
// every role winds down, outstanding copies and MMAs are drained, TMEM is
// freed and the partition is marked invalid (sum = -1, status TIMEOUT).
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <type_traits>

#include "common.cuh"
#include "kernels.h"
#include "params.h"
#include "plan.cuh"
#include "tc_ptx.cuh"
#include "verify_attn_e4m3.h"

namespace vae4 {

struct TcArgs {
  long long wait_limit;   // SM cycles before a pipeline wait gives up
  long long drain_limit;  // SM cycles the wind-down waits for copies and MMAs in flight
  int32_t n_rg;          // row groups per KV head
};

template <int D, int N, bool HL = false>
struct TcCfg {
  static_assert(N % 16 == 0 && N >= 16 && N <= 64, "rows per CTA");
  static constexpr int NSW = 8;                 // softmax warps
  static constexpr int NC = N / 2;              // rows per softmax thread
  static constexpr int IB = D < 128 ? D : 128;  // TMA box inner bytes
  static constexpr int NDH = D / IB;            // boxes per key row
  static constexpr int SMASK = IB == 128 ? 7 : 3;     // 128B / 64B swizzle
  static constexpr int DB = D / 64 < 2 ? 2 : D / 64;  // 64-d blocks of V^T (D=64 padded)
  static constexpr int MH = DB / 2;             // 128-row M halves of V^T.P^T
  static constexpr int SC = (N + 31) / 32 * 32; // TMEM columns per accumulator
  // groups of the TMEM K tile released one by one to the next tile's
  // decode: two (128-d halves) for N = 16; with more rows the softmax and
  // value chains are as long as the K chain, and the overlap (whose TMEM
  // stores slow the MMA issue, and each release costs a commit) measured
  // slower with 2 or 4 groups
  static constexpr int KFG = (N <= 16 && D >= 128) ? 2 : 1;
  // TMEM columns: K (128 keys x D/2), two S^T buffers, O^T, then the V^T
  // half-tile ring (lane = d of a 128-d block, 32 columns per block)
  static constexpr int KCOL = 0, SCOL = 128, OCOL = 128 + 2 * SC;
  static constexpr int VCOL = OCOL + MH * SC;
  static constexpr int VTC = MH * 32;           // columns per V^T half-tile
  static constexpr int NVF = (512 - VCOL) / VTC < 4 ? (512 - VCOL) / VTC : 4;
  static constexpr int QB = (D / 64) * N * 128; // Q, K-major SW128
  static constexpr int PB = 128 * 128;          // P^T, MN-major SW128 (N <= 64)
  static constexpr int NPB = HL ? 2 : 1;        // P^T buffers: P, or P_hi and P_lo
  static constexpr int RSLOT = 64 * D;          // one raw K or V half-tile
  static constexpr int SMALL = 2880;
  static constexpr int LIMIT = 232448 - 1024;   // opt-in maximum minus alignment slack
  // raw slots: half of what shared memory is left (at most 8) for K; V,
  // consumed a chain later, gets at most 4 (NVR >= NVF keeps the V
  // decoders' slot waits unambiguous).  At D = 256 this is 5 K and 4 V
  // half-tiles: measured faster per step than 5 and 6 (the whole space),
  // and than 4/5, 5/5, 4/6, 3/6, 3/5 and 4/4.
  static constexpr int NRAW = (LIMIT - QB - NPB * PB - SMALL) / RSLOT;
  static constexpr int NKR = NRAW / 2 < 8 ? NRAW / 2 : 8;
  static constexpr int NVR = NRAW - NKR < 4 ? NRAW - NKR : 4;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_P = OFF_Q + QB;
  static constexpr int OFF_KR = OFF_P + NPB * PB;
  static constexpr int OFF_VR = OFF_KR + NKR * RSLOT;
  static constexpr int OFF_SMALL = OFF_VR + NVR * RSLOT;
  static constexpr int SMEM = OFF_SMALL + SMALL + 1024;
  static constexpr int NTHREADS = 32 * 20;
  // mbarrier indices, derived from the ring sizes so no two roles share one
  static constexpr int B_KFULL = 0, B_KEMPTY = B_KFULL + NKR, B_VFULL = B_KEMPTY + NKR,
                       B_VEMPTY = B_VFULL + NVR, B_KREADY = B_VEMPTY + NVR,
                       B_KFREE = B_KREADY + 1, B_VREADY = B_KFREE + KFG, B_VFREE = B_VREADY + NVF,
                       B_SFULL = B_VFREE + NVF, B_SFREE = B_SFULL + 2, B_PREADY = B_SFREE + 2,
                       B_PVDONE = B_PREADY + 1, B_DRAINQK = B_PVDONE + 1,
                       B_DRAINPV = B_DRAINQK + 1, NBARS = B_DRAINPV + 1;
  static_assert(NBARS * 8 <= 512, "barriers fit below the small-region scalars");
  static_assert(NKR <= 8 && NVR <= 8, "producer bookkeeping");
  static_assert(NKR >= 2 && NVF >= 2 && NVR >= NVF, "slot reuse order (see the decoders)");
  static_assert(VCOL + NVF * VTC <= 512, "TMEM budget");
  static_assert(SMEM <= 232448, "shared memory budget");
  static_assert(NC % 8 == 0, "softmax column groups of 8");
};

// warp roles
enum : int {
  kWSoftmax = 0,   // 0..7
  kWKDec = 8,      // 8..11 (quadrant = warp & 3)
  kWVDec = 12,     // 12..15
  kWKProd = 16, kWVProd = 17, kWQk = 18, kWPv = 19
};
// device-side plan scratch in the P^T buffer: (L, q_len) pairs of up to
// kDevPlanMaxB sequences from byte 0, the published plan at byte kPlanSh
constexpr int kPlanSh = 12288;
// offsets in the small region (the mbarriers occupy its first 512 bytes)
constexpr int kSmTslot = 512, kSmAbort = 516, kSmBad = 520, kSmCta = 544, kSmM = 576,
              kSmPos = 832, kSmMNew = 1088, kSmBase = 1344, kSmThr = 1600,
              kSmRed = 1856;  // red: 8 warps x 32 floats, ends at 2880

__device__ __forceinline__ uint32_t sw128(uint32_t off) { return off ^ (((off >> 7) & 7u) << 4); }

// Zero the raw V bytes of keys kz .. 63 of a half-tile slot in the columns
// V decoder warp dq reads (d = 128 mh + 32 dq + 0..31).  The slot was
// written by the tensor copy (async proxy) and will be again after the
// decoders release it, hence the proxy fence after the generic stores.
template <int D, int IB, int SMASK, int MH>
static __device__ __noinline__ void zero_v_tail(uint8_t *raw, int kz, int dq, int lane) {
  constexpr int NG = 2 * MH;  // 16-byte column granules of the warp per key
  for (int i = lane; i < (64 - kz) * NG; i += 32) {
    const int k = kz + i / NG, g = i % NG;
    const int dch = 128 * (g >> 1) + 32 * dq + 16 * (g & 1);
    if (dch < D) {
      const int dh = dch / IB, cc = (dch % IB) >> 4;
      const uint32_t off = (uint32_t)((k & 15) * IB + cc * 16);
      *reinterpret_cast<uint4 *>(raw + (k >> 4) * (16 * D) + dh * (16 * IB) +
                                 (off ^ (((off >> 7) & SMASK) << 4))) = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  tc::fence_proxy_async_smem();
  __syncwarp();
}

// Producer of one ring (K or V) for caches whose strides are multiples of 8
// bytes but not all of 16 (the pages' 264-byte token stride, PR #524
// "[Kernel][SM70] Add opt-in E4M3 grouped attention with FP32 partials", AI
// integration review), which no tensor map can describe: every key row of a
// half-tile arrives as 8-byte asynchronous copies into the same swizzled
// slot layout the tensor loads produce, and each lane's completion arrives
// on the slot's "full" barrier (32 arrivals per phase).  Keys past the
// partition and pages with invalid ids are zero-filled.  Out of line: the
// tensor-load producer is the hot path.  Returns the half-tiles issued.
template <int D>
static __device__ __noinline__ int cpa_produce(const SplitParams &p, int h, int k0, int k1,
                                               int nhalf, bool isv, uint32_t ring, uint32_t full0,
                                               uint32_t empty0, int nslot, volatile int *abort_f,
                                               long long lim, volatile int *bad_f, int cur,
                                               int nxt, int lp_base, const int32_t *btb,
                                               int lane) {
  constexpr int IB = D < 128 ? D : 128, SMASK = IB == 128 ? 7 : 3;
  constexpr int CPK = D / 8, KPI = 32 / CPK;  // 8-byte chunks per key, keys per instruction
  constexpr int RSLOT = 64 * D;
  const uint8_t *hbase = (isv ? p.v_base : p.k_base) + (int64_t)h * (isv ? p.v_hs : p.k_hs);
  const int64_t ps = isv ? p.v_ps : p.k_ps, ts = isv ? p.v_ts : p.k_ts;
  const uint64_t pol = tc::l2_evict_first_policy();
  const int c = lane % CPK, kk = lane / CPK;
  const int dh = (8 * c) / IB, cb = (8 * c) % IB;  // this lane's chunk: IB block, byte in it
  const int ppb = p.page >> 4;
  const int box0 = (k0 >> 4) + lane;  // lane g < 4: box g of the first half-tile
  int lpg = box0 / ppb, sbg = box0 - lpg * ppb;
  int st = 0, u = 0, n_issued = 0;
  for (int t = 0; t < nhalf; ++t) {
    if (u > 0 && !tc::mbar_wait(empty0 + 8u * st, (u - 1) & 1, abort_f, lim)) break;
    n_issued = t + 1;
    const int rel = lpg - lp_base;
    const int pc = __shfl_sync(0xffffffffu, cur, rel & 31);
    const int pn = __shfl_sync(0xffffffffu, nxt, rel & 31);
    int phys = -1;  // lanes 0-3: page of box `lane`, -1 = zero fill
    if (lane < 4 && k0 + 64 * t + 16 * lane < k1) {
      const int ph = rel < 32 ? pc : pn;
      if (ph >= 0 && ph < p.n_pages)
        phys = ph;
      else
        *bad_f = 1;
    }
    const uint32_t slot = ring + st * RSLOT;
#pragma unroll 1
    for (int g = 0; g < 4; ++g) {
      const int pg = __shfl_sync(0xffffffffu, phys, g);
      const int sb = __shfl_sync(0xffffffffu, sbg, g);
      const int key0 = k0 + 64 * t + 16 * g;  // first key of box g
      const uint8_t *src = hbase + (int64_t)max(pg, 0) * ps + (int64_t)(16 * sb + kk) * ts + 8 * c;
#pragma unroll
      for (int r = kk; r < 16; r += KPI) {
        const bool ok = pg >= 0 && key0 + r < k1;
        const uint32_t off = (uint32_t)(r * IB + cb);
        tc::cp_async8_hint(slot + g * (16 * D) + dh * (16 * IB) + (off ^ (((off >> 7) & SMASK) << 4)),
                           ok ? src : hbase, ok ? 8 : 0, pol);
        src += KPI * ts;
      }
    }
    tc::cp_async_mbar_arrive_noinc(full0 + 8u * st);
    if (ppb == 1) {
      lpg += 4;
    } else {
      sbg += 4;
      while (sbg >= ppb) {
        sbg -= ppb;
        ++lpg;
      }
    }
    if (__shfl_sync(0xffffffffu, lpg, 0) >= lp_base + 32) {  // slide the window
      cur = nxt;
      lp_base += 32;
      const int lp = lp_base + 32 + lane;
      nxt = lp < p.max_pages ? __ldg(btb + lp) : -1;
    }
    if (++st == nslot) {
      st = 0;
      ++u;
    }
  }
  return n_issued;
}

// Partition plans, one instantiation each so none carries another's code:
// kPlanFixed: static grid (partition, head x row group, sequence), T given;
// kPlanFromLen: static grid, T from each sequence's length (the automatic
// plan of one sequence); kPlanDevice: the device-side balanced plan
// (grid.x = partition number, grid.y = row group).
enum { kPlanFixed = 0, kPlanFromLen = 1, kPlanDevice = 2 };
template <int D, int N, int MODE, bool HL>
__global__ void __launch_bounds__(TcCfg<D, N, HL>::NTHREADS, 1)
    split_tc_kernel(const SplitParams p, const TcArgs a, const __grid_constant__ CUtensorMap tmap_k,
                    const __grid_constant__ CUtensorMap tmap_v) {
  using C = TcCfg<D, N, HL>;
  constexpr int kKFull = C::B_KFULL, kKEmpty = C::B_KEMPTY, kVFull = C::B_VFULL,
                kVEmpty = C::B_VEMPTY, kKReady = C::B_KREADY, kKFree = C::B_KFREE,
                kVReady = C::B_VREADY, kVFree = C::B_VFREE, kSFull = C::B_SFULL,
                kSFree = C::B_SFREE, kPReady = C::B_PREADY, kPvDone = C::B_PVDONE,
                kDrainQk = C::B_DRAINQK, kDrainPv = C::B_DRAINPV;
  extern __shared__ uint8_t smem_raw[];
  const float kInf = __int_as_float(0x7f800000);
  constexpr float kLog2e = 1.4426950408889634f;
  // lazy-rescale threshold (log2 units): the running max is raised only when
  // a score exceeds it by more than 2^12, so P <= 4096 (far inside FP16).
  // Each raise costs a wait for the previous value MMA and a TMEM rescale of
  // O^T; with 30-sigma outliers 2^8 cost 3 us per step on the long q8 step,
  // 2^12 leaves 0.6 us, at a relative L2 error of 2.5e-4 instead of 2.2e-4
  // against the FP64 oracle (a wider P range inside each MMA).
  // With the high/residual split of P (HL) the value product runs on P
  // scaled by 2^11 (see the softmax), and 2^(4 + 11) keeps it inside FP16.
  constexpr float kTau = HL ? 4.0f : 12.0f;
  // HL: P' = 2^11 p is split into P_hi = fp16(P') and P_lo = fp16(P' -
  // P_hi), i.e. the residual of fp16(p) multiplied by 2^11 (PR #524
  // "[Kernel][SM70] Add opt-in E4M3 grouped attention with FP32 partials",
  // Historical R6 purpose and evidence, Scope and non-duplication); both go
  // through the value product into the same FP32 accumulator, and the exact
  // 2^-11 is applied to O and l in the epilogue.
  constexpr float kHiLoExp = HL ? 11.0f : 0.0f;

  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t sbase = (raw_addr + 1023u) & ~1023u;
  uint8_t *gbase = smem_raw + (sbase - raw_addr);
  const uint32_t sQ = sbase + C::OFF_Q, sP = sbase + C::OFF_P, sKR = sbase + C::OFF_KR,
                 sVR = sbase + C::OFF_VR, sSm = sbase + C::OFF_SMALL;
  uint8_t *gQ = gbase + C::OFF_Q, *gP = gbase + C::OFF_P, *gKR = gbase + C::OFF_KR,
          *gSm = gbase + C::OFF_SMALL;
  auto bar = [&](int i) -> uint32_t { return sSm + 8u * (uint32_t)i; };
  volatile int *abort_f = reinterpret_cast<volatile int *>(gSm + kSmAbort);
  volatile int *bad_f = reinterpret_cast<volatile int *>(gSm + kSmBad);
  float *m_s = reinterpret_cast<float *>(gSm + kSmM);      // running max (log2 units)
  int *pos_s = reinterpret_cast<int *>(gSm + kSmPos);      // last visible key per row
  float *mnew_s = reinterpret_cast<float *>(gSm + kSmMNew);
  float *base_s = reinterpret_cast<float *>(gSm + kSmBase);  // m, or 0 while m = -inf
  float *thr_s = reinterpret_cast<float *>(gSm + kSmThr);    // (m + tau) / alpha
  float *red = reinterpret_cast<float *>(gSm + kSmRed);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool producer = warp == kWKProd || warp == kWVProd;

  // ---- set-up that touches only this CTA's shared memory and TMEM, done
  // before the grid dependency wait so it overlaps the previous kernel's
  // tail: barriers, TMEM columns.
  if (tid == 0) {
    // arrival counts: TMA (expect_tx) and MMA commits arrive once; a K
    // half-tile is consumed by 2 decoder warps, a V half-tile by 4; K for a
    // tile comes from 4.
    for (int i = 0; i < C::NBARS; ++i) {
      uint32_t cnt = 1;
      if (i >= kKEmpty && i < kKEmpty + C::NKR)
        cnt = 64;
      else if (i == kKReady || (i >= kVEmpty && i < kVEmpty + C::NVR) ||
               (i >= kVReady && i < kVReady + C::NVF))
        cnt = 128;
      else if ((i >= kSFree && i < kSFree + 2) || i == kPReady)
        cnt = 32 * C::NSW;
      else if (p.kv_cpasync && ((i >= kKFull && i < kKFull + C::NKR) ||
                                (i >= kVFull && i < kVFull + C::NVR)))
        cnt = 32;  // one arrival per producer lane (8-byte copies)
      tc::mbar_init(bar(i), cnt);
    }
    *abort_f = 0;
    *bad_f = 0;
  }
  if (producer && lane == 0 && !p.kv_cpasync)  // kernel parameters
    tc::prefetch_tensormap(warp == kWVProd ? &tmap_v : &tmap_k);
  if (warp == kWQk) {
    tc::tmem_alloc(sSm + kSmTslot, 512);
    tc::tmem_relinquish();
  }
  tc::mbar_fence_init();
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tbase = *reinterpret_cast<volatile uint32_t *>(gSm + kSmTslot);
  // a CTA with nothing to do returns its TMEM columns before it exits (the
  // conditions below are the same for all of its threads)
  auto leave = [&]() {
    if (warp == kWQk) tc::tmem_dealloc(tbase, 512);
  };
  // launched as a programmatic dependent: everything below may read what the
  // previous kernel on the stream wrote (inputs) or overwrite what it reads
  // (the workspace), so wait for it to finish first.  (Global reads before
  // this point would also queue behind the previous kernel's stream.)
  asm volatile("griddepcontrol.wait;\n" ::: "memory");

  // ---- which partition: static grid (partition, head x row group,
  // sequence) or the device-side plan (grid.x = partition number, grid.y =
  // row group).
  // producers: first block-table window, requested as early as possible.
  // Lane l holds logical page lp_base + l (cur) and lp_base + 32 + l (nxt);
  // entries past the row are -1, entries past the sequence are loaded but
  // never used.
  int part, b, h, T, L, ql;
  int cur = -1, nxt = -1, lp_base = 0;
  const int32_t *btb = p.bt;
  auto fetch = [&](int lp) -> int { return lp < p.max_pages ? __ldg(btb + lp) : -1; };
  auto fetch_bt = [&](int bb, int k0_) {
    if (producer) {
      btb = p.bt + (int64_t)bb * p.bt_sb;
      lp_base = k0_ / p.page;  // any page size that is a multiple of 16
      cur = fetch(lp_base + lane);
      nxt = fetch(lp_base + 32 + lane);
    }
  };
  if constexpr (MODE == kPlanDevice) {
    // The plan needs the lengths first; meanwhile the producers fetch the
    // block-table window of the plan for every sequence at the launch
    // capacity with Qmax queries (host-computed W and partitions per
    // stream), which is the plan whenever the lengths are the capacity, and
    // fetch again if not.
    // (at the capacity every sequence keeps the same row groups, so CTA c
    // serves partition c mod the plan's partition count)
    const int npg = p.plan_np_guess;
    const int xg = (int)(blockIdx.x % (unsigned)(p.B * p.Hkv * npg));
    const int xs = xg / npg;  // stream of the guess
    const int bg = xs / p.Hkv, k0g = (xg - xs * npg) * p.plan_W_guess;
    if (bg < p.B) fetch_bt(bg, k0g);
    // The K producer warp evaluates the plan and passes it on through the
    // P^T buffer, unused until the first tile: the (L, q_len) pairs of the
    // batch staged at its start, then b, h, p, W, L and q_len of sequence b
    // at kPlanSh; the CTA's partition number (workspace slot) and row group
    // go to the small region for the epilogue.
    static_assert(C::PB >= kPlanSh + 64 && 2 * 4 * kDevPlanMaxB <= kPlanSh, "plan scratch");
    int *plan_ls = reinterpret_cast<int *>(gP);
    volatile int *plan_sh = reinterpret_cast<volatile int *>(gP + kPlanSh);
    if (warp == kWKProd) {
      const PlanIn pin{p.seq, p.seq_sb, p.seq_has_qlen, p.Qmax, p.capacity, p.B, p.Hkv,
                       p.plan_G, p.G, N};
      plan_stage(pin, plan_ls, lane);
      volatile int *xr = reinterpret_cast<volatile int *>(gSm + kSmCta);
      const PlanCta c = plan_cta(pin, plan_ls, blockIdx.x, lane, xr);
      if (lane == 0) {
        plan_sh[0] = c.b;
        plan_sh[1] = c.h;
        plan_sh[2] = c.p;
        plan_sh[3] = c.W;
        plan_sh[4] = c.p >= 0 ? plan_ls[2 * c.b] : 0;
        plan_sh[5] = c.p >= 0 ? plan_ls[2 * c.b + 1] : 0;
        // the stream's first slot and partition count, for the combine
        if (c.p == 0 && xr[1] == 0) p.plan_tab[c.b * p.Hkv + c.h] = make_int2(xr[0], c.np);
      }
    }
    __syncthreads();
    b = plan_sh[0];
    h = plan_sh[1];
    part = plan_sh[2];
    T = plan_sh[3];
    L = plan_sh[4];
    ql = plan_sh[5];
    if (part < 0)
      b = h = part = L = ql = 0;  // past the plan: leaves below as a dead partition
    else if (b != bg || part * T != k0g)
      fetch_bt(b, part * T);  // not the guessed partition
  } else {
    part = blockIdx.x;
    b = blockIdx.z;
    h = blockIdx.y / a.n_rg;
    T = p.T;
    if constexpr (MODE != kPlanFromLen) fetch_bt(b, part * T);  // in flight with the length reads
    L = p.seq[(int64_t)b * p.seq_sb];
    ql = p.seq_has_qlen ? p.seq[(int64_t)b * p.seq_sb + 1] : p.Qmax;
    if constexpr (MODE == kPlanFromLen) {
      // the sequence's P partitions share its L tokens; the block table is
      // read once the length is known (fetching the window of the plan at
      // the capacity first, with a second fetch on a miss, measured no
      // earlier first data and a slightly slower kernel)
      if (L > 0 && L <= p.capacity) T = max(64, plan_t_from_len(L, p.P));
      fetch_bt(b, part * T);
    }
  }
  // row group and workspace slot: from the CTA index (static grids) or
  // the plan's values in shared memory (device plan; the address is
  // recomputed from the symbol where they are read), cheap to fetch again
  // where they are needed, in the epilogue
  constexpr bool DEV = MODE == kPlanDevice;
  auto cta_sm = [&]() -> uint32_t {
    return ((smem_u32(smem_raw) + 1023u) & ~1023u) + C::OFF_SMALL + kSmCta;
  };
  auto cta_rg = [&]() -> int {
    return DEV ? tc::ld_shared_s32(cta_sm() + 4) : (int)(blockIdx.y % a.n_rg);
  };
  auto cta_slot = [&]() -> int64_t {
    return DEV ? (int64_t)tc::ld_shared_s32(cta_sm())
               : ((int64_t)blockIdx.z * p.Hkv + blockIdx.y / a.n_rg) * p.P + blockIdx.x;
  };
  const int row0 = cta_rg() * N;  // first row of this CTA's row group

  // ---- sequence, partition
  if (L < 0 || L > p.capacity) {
    if (part == 0 && blockIdx.y == 0 && tid == 0) atomicOr(p.status, VAE4_STATUS_BAD_LENGTH);
    leave();
    return;
  }
  if (ql < 0 || ql > p.Qmax || (L > 0 && ql > L)) {
    if (part == 0 && blockIdx.y == 0 && tid == 0) atomicOr(p.status, VAE4_STATUS_BAD_QLEN);
    leave();
    return;
  }
  const int k0 = part * T;
  // dead partition, or a row group whose rows are all past q_len (its
  // queries are padding: the combine writes those rows as zeros)
  if (k0 >= L || row0 >= ql * p.G) {
    leave();
    return;
  }
  const int k1 = min(k0 + T, L);
  const int ntiles = (k1 - k0 + 127) >> 7;
  const int nhalf = 2 * ntiles;  // half-tiles, the last may be all padding

  const long long LIM = a.wait_limit;
  // the combine kernel may be placed on SMs as they free up; it waits for
  // this grid's completion before reading any partial
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  // ---- queries and per-row state (everyone but the producers)
  constexpr int kSetup = C::NTHREADS - 64;  // every thread but the producers
  if (!producer) {
    const int st_id = tid < 32 * kWKProd ? tid : tid - 64;
    const __half *qb = static_cast<const __half *>(p.q) + (int64_t)b * p.q_sb;
    constexpr int QCH = D / 8;  // 16-byte chunks per query row
    for (int c = st_id; c < N * QCH; c += kSetup) {
      const int r = c / QCH, cc = c - r * QCH;
      const int rr = row0 + r, i = rr / p.G, g = rr - i * p.G;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (rr < p.rows && i < ql)
        v = __ldg(reinterpret_cast<const uint4 *>(qb + (int64_t)i * p.q_si +
                                                  (int64_t)(h * p.G + g) * p.q_sh + cc * 8));
      const int katom = cc >> 3, c8 = cc & 7;
      *reinterpret_cast<uint4 *>(gQ + katom * (N * 128) + sw128(r * 128 + c8 * 16)) = v;
    }
    for (int r = st_id; r < N; r += kSetup) {
      const int rr = row0 + r, i = rr / p.G;
      pos_s[r] = (rr < p.rows && i < ql) ? L - ql + i : -1;
      m_s[r] = -kInf;
      base_s[r] = 0.f;
      thr_s[r] = -kInf;
    }
    tc::fence_proxy_async_smem();  // Q is read by the tensor core
    tc::named_bar(2, kSetup);
  }

  int n_issued = 0;        // producers: half-tiles issued
  bool mma_issued = false;    // this thread issued tcgen05.mma

  if (producer) {
    // =============================== producers (K ring, V ring)
    // Per half-tile, lanes 0-3 each issue one 16-key box (one page slice)
    // in the same instruction.  Each lane keeps the (page, box-in-page) of
    // its box and advances it by 4 boxes per half-tile: no division in the
    // loop, whose length paces the whole stream.
    const bool isv = warp == kWVProd;
    const int nslot = isv ? C::NVR : C::NKR;
    const int fullb = isv ? kVFull : kKFull, emptyb = isv ? kVEmpty : kKEmpty;
    const uint32_t ring = isv ? sVR : sKR;
    // the KV stream is read once: keep it from pushing other data (the
    // partials the combine reads, the block table) out of L2
    const uint64_t pol = tc::l2_evict_first_policy();
    const int ppb = p.page >> 4;        // 16-key boxes per page
    const int box0 = (k0 >> 4) + lane;  // lane g < 4: box g of the first half-tile
    int lpg = box0 / ppb, sbg = box0 - lpg * ppb;
    const CUtensorMap *map = isv ? &tmap_v : &tmap_k;
    int st = 0, u = 0;  // ring slot and pass of half-tile t (t = u * nslot + st)
    if (p.kv_cpasync)
      n_issued = cpa_produce<D>(p, h, k0, k1, nhalf, isv, ring, bar(fullb), bar(emptyb), nslot,
                                abort_f, LIM, bad_f, cur, nxt, lp_base, btb, lane);
    // V, consumed a chain after K, starts ~0.6 us later (a fixed pause),
    // so K's first tile lands sooner (long step -0.2 us, ragged split -0.4)
    if (isv && !p.kv_cpasync) {
      const long long t0 = clock64();
      while (clock64() - t0 < 1200) {
      }
    }
    for (int t = 0; t < (p.kv_cpasync ? 0 : nhalf); ++t) {
      if (u > 0 && !tc::mbar_wait(bar(emptyb + st), (u - 1) & 1, abort_f, LIM)) break;
      if (lane == 0) tc::mbar_arrive_expect_tx(bar(fullb + st), C::RSLOT);
      n_issued = t + 1;
      // block-table window: lane 0's page is in [lp_base, lp_base + 32) and
      // the others' at most 3 pages on, so every box finds its id in cur/nxt
      const int rel = lpg - lp_base;
      const int pc = __shfl_sync(0xffffffffu, cur, rel & 31);
      const int pn = __shfl_sync(0xffffffffu, nxt, rel & 31);
      if (lane < 4) {
        const int phys = rel < 32 ? pc : pn;
        int pgc = (int)p.n_pages;  // outside the tensor: zero fill
        if (k0 + 64 * t + 16 * lane < k1) {
          if (phys >= 0 && phys < p.n_pages)
            pgc = phys;
          else
            *bad_f = 1;
        }
        // one box: 16 keys x D bytes of head h, as NDH blocks of 16 x IB
        // (swizzled); coordinates (byte, token in page, block, head, page)
        tc::tma_load_5d_hint(ring + st * C::RSLOT + lane * (16 * D), map, 0, 16 * sbg, 0, h, pgc,
                             bar(fullb + st), pol);
      }
      if (ppb == 1) {
        lpg += 4;
      } else {
        sbg += 4;
        while (sbg >= ppb) {
          sbg -= ppb;
          ++lpg;
        }
      }
      if (__shfl_sync(0xffffffffu, lpg, 0) >= lp_base + 32) {  // slide the window
        cur = nxt;
        lp_base += 32;
        nxt = fetch(lp_base + 32 + lane);
      }
      // static plans: the first tile's copies go out ~0.6 us ahead of the
      // rest of the ring, so they are not queued behind every CTA's whole
      // initial burst (a fixed pause, no condition: measured -0.2 us on the
      // long step and -0.4 us on tp4; slower with the device plan)
      if (MODE != kPlanDevice && t == 1) {
        const long long t0 = clock64();
        while (clock64() - t0 < 1200) {
        }
      }
      if (++st == nslot) {
        st = 0;
        ++u;
      }
    }
  } else if (warp == kWQk) {
    // =============================== score MMA issuer: S^T = K . Q^T
    if (lane == 0) {
      constexpr uint32_t id_qk = tc::idesc_f16(128, N, 0, 0);
      for (int j = 0; j < ntiles; ++j) {
        if (!tc::mbar_wait(bar(kKReady), j & 1, abort_f, LIM)) break;
        if (j >= 2 && !tc::mbar_wait(bar(kSFree + (j & 1)), ((j >> 1) - 1) & 1, abort_f, LIM))
          break;
        tc::tc_fence_after();
        const uint32_t d = tbase + C::SCOL + (j & 1) * C::SC;
        constexpr int MPG = D / 16 / C::KFG;  // MMAs per released group
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t bq = sQ + (ks >> 2) * (N * 128) + (ks & 3) * 32;
          tc::mma_ts(d, tbase + C::KCOL + ks * 8, tc::smem_desc(bq, 16, 1024), id_qk, ks > 0);
          if constexpr (C::KFG > 1)
            if ((ks + 1) % MPG == 0) tc::mma_commit(bar(kKFree + ks / MPG));
        }
        tc::mma_commit(bar(kSFull + (j & 1)));
        if constexpr (C::KFG == 1) tc::mma_commit(bar(kKFree));
        mma_issued = true;
      }
    }
  } else if (warp == kWPv) {
    // =============================== value MMA issuer: O^T += V^T . P^T
    if (lane == 0) {
      constexpr uint32_t id_pv = tc::idesc_f16(128, N, 0, 1);
      bool ok = true;
      for (int j = 0; ok && j < ntiles; ++j) {
        if (!(ok = tc::mbar_wait(bar(kPReady), j & 1, abort_f, LIM))) break;
        for (int kh = 0; kh < 2 && ok; ++kh) {
          const int t = 2 * j + kh, vs = t % C::NVF;
          if (!(ok = tc::mbar_wait(bar(kVReady + vs), (t / C::NVF) & 1, abort_f, LIM))) break;
          tc::tc_fence_after();
#pragma unroll
          for (int mh = 0; mh < C::MH; ++mh) {
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4) {
              const int ks = kh * 4 + k4;
              const uint32_t av = tbase + C::VCOL + vs * C::VTC + mh * 32 + k4 * 8;
              const uint32_t bp = sP + ks * 2048;
              tc::mma_ts(tbase + C::OCOL + mh * C::SC, av, tc::smem_desc(bp, 16384, 1024), id_pv,
                         (j > 0 || ks > 0) ? 1u : 0u);
              if constexpr (HL)  // the residual, same V^T, same accumulator
                tc::mma_ts(tbase + C::OCOL + mh * C::SC, av,
                           tc::smem_desc(bp + C::PB, 16384, 1024), id_pv, 1u);
            }
          }
          tc::mma_commit(bar(kVFree + vs));
          mma_issued = true;
        }
        if (!ok) break;
        tc::mma_commit(bar(kPvDone));
      }
    }
  } else if (warp >= kWKDec && warp < kWVDec) {
    // =============================== K decoders (thread = key)
    const int dq = warp & 3;              // TMEM lane quadrant = keys 32*dq.. of a tile
    const int kh = dq >> 1;               // half-tile of the 128-key tile
    const int kk = 32 * (dq & 1) + lane;  // key within the half-tile
    const uint32_t lane_off = (uint32_t)(32 * dq) << 16;
    // one copy of the loop per KV format (the run takes one of them)
    auto decode_k = [&](auto e5m2) {
      constexpr bool E5 = decltype(e5m2)::value;
      for (int j = 0; j < ntiles; ++j) {
        const int t = 2 * j + kh;
        // K -> TMEM: column c holds d = 2c (low half), 2c+1 (high half).
        // Wait for the previous tile's score MMAs (of the first released
        // group) first: they prove every decoder warp finished that tile,
        // hence waited for every earlier K half-tile (in particular this
        // slot's previous use, t - NKR <= t - 2), so the parity wait on the
        // slot below cannot match an older phase when pairs share slots.
        // Later groups are overwritten once their MMAs are done.
        const int st = t % C::NKR;
        if (j > 0 && !tc::mbar_wait(bar(kKFree), (j - 1) & 1, abort_f, LIM)) break;
        if (!tc::mbar_wait(bar(kKFull + st), (t / C::NKR) & 1, abort_f, LIM)) break;
        tc::tc_fence_after();
        const uint8_t *rawK = gKR + st * C::RSLOT;
        bool ok = true;
#pragma unroll
        for (int grp = 0; grp < D / 64; ++grp) {
          if constexpr (C::KFG > 1) {
            if (grp > 0 && j > 0) {
              if (!(ok = tc::mbar_wait(bar(kKFree + grp * C::KFG / (D / 64)), (j - 1) & 1,
                                       abort_f, LIM)))
                break;
              tc::tc_fence_after();
            }
          }
          uint32_t r[32];
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            const int c = grp * 4 + q4;  // 16-byte chunk of the key row
            const int dh = (c * 16) / C::IB, cc = ((c * 16) % C::IB) >> 4;
            const uint32_t off = (uint32_t)((kk & 15) * C::IB + cc * 16);
            const uint4 w = *reinterpret_cast<const uint4 *>(
                rawK + (kk >> 4) * (16 * D) + dh * (16 * C::IB) +
                (off ^ (((off >> 7) & C::SMASK) << 4)));
            const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              r[q4 * 8 + 2 * e] = fp8x2_to_f16x2<E5>(wv[e]);
              r[q4 * 8 + 2 * e + 1] = fp8x2_to_f16x2<E5>(wv[e] >> 16);
            }
          }
          const uint32_t (&r0)[16] = *reinterpret_cast<const uint32_t(*)[16]>(&r[0]);
          const uint32_t (&r1)[16] = *reinterpret_cast<const uint32_t(*)[16]>(&r[16]);
          tc::tmem_st16(tbase + lane_off + C::KCOL + grp * 32, r0);
          tc::tmem_st16(tbase + lane_off + C::KCOL + grp * 32 + 16, r1);
        }
        if (!ok) break;
        tc::tmem_wait_st();
        tc::tc_fence_before();
        tc::mbar_arrive(bar(kKReady));
        tc::mbar_arrive(bar(kKEmpty + st));
      }
    };
    if (p.kv_e5m2)
      decode_k(std::true_type{});
    else
      decode_k(std::false_type{});
  } else if (warp >= kWVDec && warp < kWKProd) {
    // =============================== V decoders (warp = 32 d per 128-d block)
    const int dq = warp & 3;  // TMEM lane quadrant = d 32*dq.. of each 128-d block
    // ldmatrix rows: threads 0-15 give keys 0-15 of a page, 16-31 the same
    // rows of the next page (two 16 x 16 byte matrices per load)
    const int pr = lane & 15, pg = lane >> 4;
    auto decode_v = [&](auto e5m2) {
      constexpr bool E5 = decltype(e5m2)::value;
      for (int t = 0; t < nhalf; ++t) {
        // V -> V^T in TMEM (lane = d, column c = keys 2c, 2c+1).  Wait for
        // the value MMA that last read the V^T slot first: it proves
        // half-tiles up to t - NVF >= t - NVR were decoded, i.e. this raw
        // slot's previous use is complete, so the parity wait below is
        // unambiguous.
        const int st = t % C::NVR, vs = t % C::NVF;
        if (t >= C::NVF && !tc::mbar_wait(bar(kVFree + vs), ((t / C::NVF) - 1) & 1, abort_f, LIM))
          break;
        if (!tc::mbar_wait(bar(kVFull + st), (t / C::NVR) & 1, abort_f, LIM)) break;
        tc::tc_fence_after();
        const uint32_t rawV = sVR + st * C::RSLOT;
        // The box holding key k1 - 1 is loaded whole, so up to 15 of its
        // keys lie past the partition.  When k1 = L those pool slots may
        // never have been written (a NaN or infinity code there would turn
        // the masked key's P = 0 into a NaN product): this warp zeroes its
        // columns of those keys (boxes that start at or past k1 are
        // zero-filled by the copy itself).  Out of line, so the hot loop
        // below keeps its code.
        const int kz = k1 - k0 - 64 * t;  // keys of the half-tile before k1
        if (kz > 0 && kz < 64 && (kz & 15) != 0)
          zero_v_tail<D, C::IB, C::SMASK, C::MH>(gbase + C::OFF_VR + st * C::RSLOT, kz, dq, lane);
#pragma unroll
        for (int mh = 0; mh < C::MH; ++mh) {
#pragma unroll
          for (int dc = 0; dc < 2; ++dc) {
            const int dch = 128 * mh + 32 * dq + 16 * dc;  // first d of the 16-d chunk
            if (dch < D) {
              const int dh = dch / C::IB, cc = (dch % C::IB) >> 4;
              const uint32_t off = (uint32_t)(pr * C::IB + cc * 16);
              const uint32_t src = rawV + dh * (16 * C::IB) + (off ^ (((off >> 7) & C::SMASK) << 4));
#pragma unroll
              for (int kp = 0; kp < 2; ++kp) {  // keys 32 kp .. 32 kp + 31
                uint32_t m4[4];
                ldsm_b8_trans_x2(m4, src + (2 * kp + pg) * (16 * D));
                // m4[0]: keys 4(l%4) + 0..3 of d = l/4, m4[1]: of d + 8;
                // m4[2], m4[3]: the same for the keys 16 later
                uint32_t v[8];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  v[2 * e] = fp8x2_to_f16x2<E5>(m4[e]);
                  v[2 * e + 1] = fp8x2_to_f16x2<E5>(m4[e] >> 16);
                }
                tc::tmem_st_16x256b_x2(tbase + ((uint32_t)(32 * dq + 16 * dc) << 16) + C::VCOL +
                                           vs * C::VTC + mh * 32 + kp * 16,
                                       v);
              }
            }
          }
        }
        tc::tmem_wait_st();
        tc::tc_fence_before();
        tc::mbar_arrive(bar(kVReady + vs));
        tc::mbar_arrive(bar(kVEmpty + st));
      }
    };
    if (p.kv_e5m2)
      decode_v(std::true_type{});
    else
      decode_v(std::false_type{});
  } else if (warp < kWKDec) {
    // =============================== softmax (thread = key, NC rows)
    const int q = warp & 3, cg = warp >> 2;
    const int col0 = cg * C::NC;
    const uint32_t lane_off = (uint32_t)(32 * q) << 16;
    // K holds dec(b) exactly; t = S * alpha is the score in log2 units
    const float alpha = p.sm_scale * p.scales[h * p.scale_sh] * kLog2e;
    // every real row sees keys 0 .. L - q_len; padding rows have zero
    // queries (finite, never output), so only tiles past that key or past
    // the partition end need the per-row mask
    const int min_pos = L - ql;
    constexpr int nsm = 32 * C::NSW;
    float lpart[C::NC];
#pragma unroll
    for (int c = 0; c < C::NC; ++c) lpart[c] = 0.f;
    bool alive = true;
    for (int j = 0; j < ntiles; ++j) {
      const int buf = j & 1;
      float s[C::NC];
      alive = alive && tc::mbar_wait(bar(kSFull + buf), (j >> 1) & 1, abort_f, LIM);
      if (alive) {
        tc::tc_fence_after();
#pragma unroll
        for (int c8 = 0; c8 < C::NC / 8; ++c8) {
          uint32_t r[8];
          tc::tmem_ld8(tbase + lane_off + C::SCOL + buf * C::SC + col0 + c8 * 8, r);
#pragma unroll
          for (int e = 0; e < 8; ++e) s[c8 * 8 + e] = __uint_as_float(r[e]);
        }
        tc::tmem_wait_ld();
        tc::tc_fence_before();
      } else {
#pragma unroll
        for (int c = 0; c < C::NC; ++c) s[c] = 0.f;
      }
      tc::mbar_arrive(bar(kSFree + buf));

      const int key = k0 + 128 * j + 32 * q + lane;
      bool exceed = false;
      if (key < k1 && key <= min_pos) {
#pragma unroll
        for (int c = 0; c < C::NC; ++c) exceed |= s[c] > thr_s[col0 + c];
      } else {
        const bool kvalid = key < k1;
#pragma unroll
        for (int c = 0; c < C::NC; ++c) {
          s[c] = (kvalid && key <= pos_s[col0 + c]) ? s[c] : -kInf;
          exceed |= s[c] > thr_s[col0 + c];
        }
      }
      // did any score of the tile exceed its row's threshold (all softmax warps)
      const bool any = tc::named_bar_or(1, nsm, exceed);
      if (any) {
        // exact tile maximum per row over the 128 keys (4 quadrant warps)
#pragma unroll
        for (int c = 0; c < C::NC; ++c) {
          float mx = s[c];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
          if (lane == 0) red[warp * 32 + c] = mx * alpha;  // -inf stays -inf
        }
        tc::named_bar(1, nsm);
        if (q == 0 && lane < C::NC) {  // one warp per column group combines the quadrants
          float mt = red[(cg * 4) * 32 + lane];
#pragma unroll
          for (int qq = 1; qq < 4; ++qq) mt = fmaxf(mt, red[(cg * 4 + qq) * 32 + lane]);
          mnew_s[col0 + lane] = fmaxf(m_s[col0 + lane], mt);
        }
        tc::named_bar(1, nsm);
        // factors 2^(m_old - m_new) for the running sums ...
#pragma unroll
        for (int c = 0; c < C::NC; ++c) {
          const float mo = m_s[col0 + c], mn = mnew_s[col0 + c];
          lpart[c] *= (mn == mo) ? 1.f : fast_exp2(mo - mn);
        }
        if (j > 0) {
          // ... and for the O^T columns, once P.V of the previous tile is done
          alive = alive && tc::mbar_wait(bar(kPvDone), (j - 1) & 1, abort_f, LIM);
          if (alive) {
            tc::tc_fence_after();
#pragma unroll
            for (int mh = 0; mh < C::MH; ++mh) {
#pragma unroll
              for (int c8 = 0; c8 < C::NC / 8; ++c8) {
                const uint32_t ta = tbase + lane_off + C::OCOL + mh * C::SC + col0 + c8 * 8;
                uint32_t r[8];
                tc::tmem_ld8(ta, r);
                tc::tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                  const float mo = m_s[col0 + c8 * 8 + e], mn = mnew_s[col0 + c8 * 8 + e];
                  const float f = (mn == mo) ? 1.f : fast_exp2(mo - mn);
                  r[e] = __float_as_uint(__uint_as_float(r[e]) * f);
                }
                tc::tmem_st8(ta, r);
              }
            }
            tc::tmem_wait_st();
          }
        }
        tc::named_bar(1, nsm);  // every thread has read the old maxima
        if (q == 0 && lane < C::NC) {
          const float mn = mnew_s[col0 + lane];
          m_s[col0 + lane] = mn;
          base_s[col0 + lane] = mn == -kInf ? 0.f : mn;
          thr_s[col0 + lane] = (mn + kTau) / alpha;
        }
        tc::named_bar(1, nsm);  // new maxima visible
      }
      // the single P buffer is free once P.V of the previous tile is done
      if (j > 0) alive = alive && tc::mbar_wait(bar(kPvDone), (j - 1) & 1, abort_f, LIM);
      // p = 2^(t - m): FP16 into P^T (MN-major, 128-byte swizzle); the row
      // sums add the same rounded values
      const int kt = 32 * q + lane;  // key within the tile
#pragma unroll
      for (int c8 = 0; c8 < C::NC / 8; ++c8) {
        uint32_t hw[4], lw[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int c = c8 * 8 + 2 * e;
          float b0 = -base_s[col0 + c], b1 = -base_s[col0 + c + 1];
          if constexpr (HL) {
            b0 += kHiLoExp;
            b1 += kHiLoExp;
          }
          const float e0 = fast_exp2(fmaf(s[c], alpha, b0));
          const float e1 = fast_exp2(fmaf(s[c + 1], alpha, b1));
          const __half2 hh = __floats2half2_rn(e0, e1);
          const float2 fl = __half22float2(hh);
          if constexpr (HL) {
            // e - fl is exact in FP32; hi + lo (22 significant bits) too
            const __half2 ll = __floats2half2_rn(e0 - fl.x, e1 - fl.y);
            const float2 fr = __half22float2(ll);
            lpart[c] += fl.x + fr.x;
            lpart[c + 1] += fl.y + fr.y;
            lw[e] = *reinterpret_cast<const uint32_t *>(&ll);
          } else {
            lpart[c] += fl.x;
            lpart[c + 1] += fl.y;
          }
          hw[e] = *reinterpret_cast<const uint32_t *>(&hh);
        }
        const int r0 = col0 + c8 * 8;
        const uint32_t po = sw128((uint32_t)(kt * 128 + (r0 >> 3) * 16));
        *reinterpret_cast<uint4 *>(gP + po) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        if constexpr (HL)
          *reinterpret_cast<uint4 *>(gP + C::PB + po) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
      }
      tc::fence_proxy_async_smem();
      tc::tc_fence_before();
      tc::mbar_arrive(bar(kPReady));
    }

    // ---- epilogue: row sums and the unnormalised O^T of this partition
#pragma unroll
    for (int c = 0; c < C::NC; ++c) {
      float sm = lpart[c];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sm += __shfl_xor_sync(0xffffffffu, sm, o);
      if (lane == 0) red[warp * 32 + c] = sm;
    }
    alive = alive && tc::mbar_wait(bar(kPvDone), (ntiles - 1) & 1, abort_f, LIM);
    tc::tc_fence_before();
  }

  // ---- O^T out of TMEM: softmax and decoder warps (4 per lane quadrant)
  // share the columns once the last value MMA is done
  if (warp < kWKProd) {
    tc::named_bar(3, 32 * kWKProd);
    tc::tc_fence_after();
    if (*abort_f == 0) {  // every softmax warp saw the last value MMA complete
      const int q = warp & 3, k4 = warp >> 2;
      constexpr int NG = C::MH * (N / 8);        // 8-column groups per lane quadrant
      constexpr int GPW = (NG + 3) / 4;          // groups per warp
      const int64_t slot = cta_slot() * p.rows_pad + cta_rg() * N;
      uint32_t r[GPW][8];
#pragma unroll
      for (int i = 0; i < GPW; ++i) {
        const int g = k4 + 4 * i;
        if (g < NG) {
          const int mh = g / (N / 8), c8 = g % (N / 8);
          tc::tmem_ld8(tbase + ((uint32_t)(32 * q) << 16) + C::OCOL + mh * C::SC + c8 * 8, r[i]);
        }
      }
      tc::tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < GPW; ++i) {
        const int g = k4 + 4 * i;
        const int mh = g / (N / 8), c8 = g % (N / 8);
        const int d = 128 * mh + 32 * q + lane;
        if (g < NG && d < D) {
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            // stored as sum p * dec(V) * 2^-8 (exact scaling): the
            // combine kernel's convention; HL also removes its 2^11
            p.ws_o[(slot + c8 * 8 + e) * D + d] =
                __uint_as_float(r[i][e]) * (HL ? 1.9073486328125e-06f : 0.00390625f);
          }
        }
      }
    }
    tc::tc_fence_before();
  }

  // ---- wind-down: drain copies and MMAs, free TMEM, publish (max, sum).
  // A run without an abort has already waited for every load and MMA it
  // issued (each was consumed); after an abort some may still be in flight.
  __syncthreads();
  const bool drain = *abort_f != 0;
  if (drain && producer && lane == 0) {
    // every issued load must have landed before the CTA's memory is released
    const int fullb = warp == kWVProd ? kVFull : kKFull;
    const int nslot = warp == kWVProd ? C::NVR : C::NKR;
    volatile int no_abort = 0;
    for (int s = 0; s < nslot && s < n_issued; ++s) {
      const int uses = (n_issued - 1 - s) / nslot + 1;  // half-tiles s, s + nslot, ...
      tc::mbar_wait(bar(fullb + s), (uses - 1) & 1, &no_abort, a.drain_limit);
    }
  }
  if (producer && p.kv_cpasync) tc::cp_async_wait_all();  // every lane's own copies
  if (drain && (warp == kWQk || warp == kWPv) && lane == 0 && mma_issued) {
    const uint32_t db = bar(warp == kWQk ? kDrainQk : kDrainPv);
    tc::mma_commit(db);
    volatile int no_abort = 0;
    tc::mbar_wait(db, 0, &no_abort, a.drain_limit);
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == kWQk) tc::tmem_dealloc(tbase, 512);
  const bool aborted = *abort_f != 0, bad = *bad_f != 0;
  if (tid == 0) {
    if (aborted) atomicOr(p.status, VAE4_STATUS_TIMEOUT);
    if (bad) atomicOr(p.status, VAE4_STATUS_BAD_BLOCK);
  }
  if (tid < N) {
    const int r = tid, cg = r / C::NC, c = r - cg * C::NC;
    float l = 0.f;
#pragma unroll
    for (int qq = 0; qq < 4; ++qq) l += red[(cg * 4 + qq) * 32 + c];
    if constexpr (HL) l *= 4.8828125e-04f;  // 2^-11, exact
    const int64_t slot = cta_slot() * p.rows_pad + cta_rg() * N;
    p.ws_ml[(slot + r) * 2 + 0] = m_s[r];
    p.ws_ml[(slot + r) * 2 + 1] = (aborted || bad) ? -1.f : l;
  }
}

// ---------------------------------------------------------------------------
// Host side: launch of one instantiation.
template <int D, int N, int MODE, bool HL>
cudaError_t launch_tc(const SplitParams &p, const TcArgs &a, const CUtensorMap &map_k,
                      const CUtensorMap &map_v, cudaStream_t stream) {
  using C = TcCfg<D, N, HL>;
  // the shared-memory opt-in is a function attribute of the device's
  // context: set it once per context (a context made after cudaDeviceReset
  // starts without it)
  constexpr int kDevs = 64;
  static std::atomic<unsigned long long> configured[kDevs] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
  const unsigned long long ctx = current_context_id();
  if (dev < 0 || dev >= kDevs || ctx == 0 ||
      configured[dev].load(std::memory_order_acquire) != ctx) {
    cudaError_t e = cudaFuncSetAttribute(split_tc_kernel<D, N, MODE, HL>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < kDevs) configured[dev].store(current_context_id(), std::memory_order_release);
  }
  // programmatic dependent launch: the CTAs may be placed while the previous
  // kernel on the stream drains; the kernel waits for it before its first
  // global-memory access that depends on it
  cudaLaunchConfig_t cfg = {};
  // device plan: one CTA per live (partition, row group), numbered row
  // group by row group (plan_row_group), so the live CTAs are the first
  // ones and all start in the first wave
  cfg.gridDim = MODE == kPlanDevice ? dim3(p.plan_G, 1, 1) : dim3(p.P, p.Hkv * a.n_rg, p.B);
  cfg.blockDim = dim3(C::NTHREADS);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, split_tc_kernel<D, N, MODE, HL>, p, a, map_k, map_v);
}

// Every (head dim, padded rows) instantiation of one plan mode.
template <int MODE, bool HL>
cudaError_t launch_tc_any(const SplitParams &p, const TcArgs &a, int n, const CUtensorMap &map_k,
                          const CUtensorMap &map_v, cudaStream_t stream) {
  switch (p.D * 1000 + n) {
    case 64016: return launch_tc<64, 16, MODE, HL>(p, a, map_k, map_v, stream);
    case 64032: return launch_tc<64, 32, MODE, HL>(p, a, map_k, map_v, stream);
    case 64048: return launch_tc<64, 48, MODE, HL>(p, a, map_k, map_v, stream);
    case 64064: return launch_tc<64, 64, MODE, HL>(p, a, map_k, map_v, stream);
    case 128016: return launch_tc<128, 16, MODE, HL>(p, a, map_k, map_v, stream);
    case 128032: return launch_tc<128, 32, MODE, HL>(p, a, map_k, map_v, stream);
    case 128048: return launch_tc<128, 48, MODE, HL>(p, a, map_k, map_v, stream);
    case 128064: return launch_tc<128, 64, MODE, HL>(p, a, map_k, map_v, stream);
    case 256016: return launch_tc<256, 16, MODE, HL>(p, a, map_k, map_v, stream);
    case 256032: return launch_tc<256, 32, MODE, HL>(p, a, map_k, map_v, stream);
    case 256048: return launch_tc<256, 48, MODE, HL>(p, a, map_k, map_v, stream);
    case 256064: return launch_tc<256, 64, MODE, HL>(p, a, map_k, map_v, stream);
    default: return cudaErrorInvalidValue;
  }
}

// The other plan modes' instantiations, each compiled in a translation unit
// of its own.
cudaError_t launch_split_tc_dev(const SplitParams &p, const TcArgs &a, int n,
                                const CUtensorMap &map_k, const CUtensorMap &map_v,
                                cudaStream_t stream);
cudaError_t launch_split_tc_len(const SplitParams &p, const TcArgs &a, int n,
                                const CUtensorMap &map_k, const CUtensorMap &map_v,
                                cudaStream_t stream);

}  // namespace vae4
