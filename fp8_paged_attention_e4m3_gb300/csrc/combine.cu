// Combine kernel: merges the FP32 partition states of each output row in a
// fixed order and writes the FP16 output.
//
// For row r of (sequence b, KV head h), over the live partitions p (those
// with p*T < L and a nonzero running sum):
//     M   = max_p m_p                  (m_p in log2 units of the score)
//     w_p = 2^(m_p - M)
//     out = (sum_p w_p O_p) / (sum_p w_p l_p) * s_V * 2^8
// all in FP32, rounded once to FP16 (round to nearest even).  It is the one
// place where the FP32 partition state (max, sum, unnormalised P.V) is
// reduced, and it reduces in FP32 (PR #524 "[Kernel][SM70] Add opt-in E4M3
// grouped attention with FP32 partials", final status; PR #560 "[Bugfix]
// Use FP32 state and E4M3 defaults for DFlash2", Purpose).
// Padding query slots, dead sequences (L == 0) and sequences whose lengths
// or pages were invalid get zeros.
//
// Work decomposition: a unit is (live row, 32-wide slice of d), taken by
// one warp.  Lane = (partition group, float4 of the slice): eight lanes read
// 128 contiguous bytes of one partition's O, four groups per warp; group g
// takes partitions g, g + 4, ... in ascending order and loads their (max,
// sum) pairs itself (its eight lanes share the address).  The group sums
// are added by a fixed shuffle tree, so the summation order depends only on
// the partition count, never on scheduling: repeated runs agree bit for
// bit.  Only live units are enumerated (a prefix over the sequences' live
// rows, computed in every block from the lengths), so the warps share them
// evenly; rows without a live query are zero-filled before the grid
// dependency wait (the split kernel does not touch the output).
#include "combine_rows.cuh"
#include "common.cuh"
#include "kernels.h"
#include "plan.cuh"
#include "verify_attn_e4m3.h"

namespace vae4 {

namespace {

// Blocks of 16 warps, two per SM (at most 64 registers: four partitions
// per lane per chunk): the blocks are placed as the split kernel's CTAs
// leave their SMs; smaller blocks piled up on the first SMs to free up
// (half the SMs took every block of the long-context step), and one block
// per SM (eight partitions per lane) left each warp more units to combine
// one after another.
constexpr int kCombineThreads = 512;
constexpr int kWarps = kCombineThreads / 32;
constexpr int kCacheB = 2048;   // lengths cached in shared memory up to this batch
constexpr int kCacheTab = 2048; // device-plan stream entries cached up to this many

struct Len {
  int L, ql;
};

__device__ __forceinline__ Len read_len(const CombineParams &p, int b) {
  const int L = p.seq[(int64_t)b * p.seq_sb];
  const int ql = p.seq_has_qlen ? p.seq[(int64_t)b * p.seq_sb + 1] : p.Qmax;
  return Len{L, ql};
}

// a row (query i) of sequence b holds a live query
__device__ __forceinline__ bool live_row(const CombineParams &p, Len l, int i) {
  return l.L > 0 && l.L <= p.capacity && l.ql >= 0 && l.ql <= p.Qmax && l.ql <= l.L && i < l.ql;
}

// Static plans whose streams spread over many partitions (one sequence over
// every SM): one CTA per (output row, 64-wide slice of d), the unit combine
// of combine_rows.cuh with the whole CTA.
__global__ void __launch_bounds__(kRowThreads) combine_rows_kernel(const CombineParams p) {
  extern __shared__ __align__(16) float rsm[];
  __shared__ float red[kRowThreads / 32];
  __shared__ float4 accs[kRowGroups][kRowLanes];
  // the next kernel on the stream may be placed as this grid's CTAs leave
  // (its own grid-dependency wait still waits for this grid to finish)
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  const int nd = p.D / 64;  // d slices per row
  const int r = blockIdx.x / nd, dsl = blockIdx.x - r * nd;
  const int h = blockIdx.y, b = blockIdx.z;
  const int i = r / p.G;
  // lengths are inputs of the step, not results of the split kernel: read
  // them before waiting for it
  const int L = p.seq[(int64_t)b * p.seq_sb];
  const int ql = p.seq_has_qlen ? p.seq[(int64_t)b * p.seq_sb + 1] : p.Qmax;
  // partitions of this (sequence, KV head): slots slot0 .. slot0 + nP - 1
  const int slot0 = (b * p.Hkv + h) * p.P;
  const int T = (p.t_from_len && L > 0 && L <= p.capacity) ? max(64, plan_t_from_len(L, p.P)) : p.T;
  const bool dead = L <= 0 || L > p.capacity || ql < 0 || ql > p.Qmax || ql > L || i >= ql;
  const int nP = dead ? 0 : (L + T - 1) / T;
  const float sv = __ldg(p.scales + h * p.scale_sh + 1);  // the head's V scale (an input)
  // wait until the split kernel's partials are complete and visible
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  if (blockIdx.x == 0 && h == 0 && threadIdx.x == 0) {  // invalid lengths, once per sequence
    if (L < 0 || L > p.capacity) atomicOr(p.status, VAE4_STATUS_BAD_LENGTH);
    else if (ql < 0 || ql > p.Qmax || (L > 0 && ql > L)) atomicOr(p.status, VAE4_STATUS_BAD_QLEN);
  }
  const RowScratch sc{rsm, rsm + p.P, red, accs};
  combine_row_unit(p, b, h, r, dsl, slot0, nP, sv, threadIdx.x, 0, sc);
}

// Sequence of live unit v: the largest b with ustart[b] <= v (sequences
// without live units own an empty range and are passed over).
__device__ __forceinline__ int find_seq(const int *ustart, int nb, int v) {
  int lo = 0, hi = nb;  // ustart[lo] <= v < ustart[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (ustart[mid] <= v)
      lo = mid;
    else
      hi = mid;
  }
  return lo;
}

__global__ void __launch_bounds__(kCombineThreads, 2) combine_kernel(const CombineParams p) {
  constexpr int PG = 4;         // partition groups per warp (eight lanes each)
  constexpr int NPL = 4;        // partitions per lane per chunk
  constexpr int CH = PG * NPL;  // partitions per chunk
  extern __shared__ __align__(16) int csm[];
  __shared__ int wsum[kWarps];
  const int nb_cache = p.B <= kCacheB ? p.B : 0;
  int2 *lens = reinterpret_cast<int2 *>(csm);  // (L, q_len) per sequence
  const int ntab = (p.dev_plan && p.B * p.Hkv <= kCacheTab) ? p.B * p.Hkv : 0;
  int2 *tab = lens + nb_cache;                          // (first slot, partitions)
  int *ustart = reinterpret_cast<int *>(tab + ntab);    // first live unit per sequence
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // the next kernel on the stream may be placed as this grid's CTAs leave
  // (its own grid-dependency wait still waits for this grid to finish)
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  const int R = p.Qmax * p.G;  // rows per (sequence, KV head)
  const int S = p.D / 32;      // slices per row
  const int64_t nunits = (int64_t)p.B * p.Hkv * R * S;

  // ---- before the grid dependency wait: inputs only.  Lengths into shared
  // memory; rows without a live query zero-filled; invalid lengths reported.
  for (int b = tid; b < nb_cache; b += kCombineThreads) {
    const Len l = read_len(p, b);
    lens[b] = make_int2(l.L, l.ql);
  }
  __syncthreads();
  auto len_of = [&](int b) -> Len {
    if (b < nb_cache) return Len{lens[b].x, lens[b].y};
    return read_len(p, b);
  };
  {
    // 16 bytes (8 halves) per thread over every output row of a query slot
    // that is not live
    const int per_row = p.D / 8;
    const int64_t n = (int64_t)p.B * p.Qmax * p.Hq * per_row;
    for (int64_t x = (int64_t)blockIdx.x * kCombineThreads + tid; x < n;
         x += (int64_t)gridDim.x * kCombineThreads) {
      const int c = (int)(x % per_row);
      const int64_t rw = x / per_row;
      const int hq = (int)(rw % p.Hq);
      const int i = (int)((rw / p.Hq) % p.Qmax);
      const int b = (int)(rw / ((int64_t)p.Hq * p.Qmax));
      if (!live_row(p, len_of(b), i)) {
        __half *o = static_cast<__half *>(p.out) + (int64_t)b * p.o_sb + (int64_t)i * p.o_si +
                    (int64_t)hq * p.o_sh + 8 * c;
        *reinterpret_cast<uint4 *>(o) = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    if (blockIdx.x == 0) {  // report invalid lengths once per sequence
      for (int b = tid; b < p.B; b += kCombineThreads) {
        const Len l = len_of(b);
        if (l.L < 0 || l.L > p.capacity)
          atomicOr(p.status, VAE4_STATUS_BAD_LENGTH);
        else if (l.ql < 0 || l.ql > p.Qmax || (l.L > 0 && l.ql > l.L))
          atomicOr(p.status, VAE4_STATUS_BAD_QLEN);
      }
    }
  }
  // Live units only, numbered sequence by sequence (KV head, row, slice
  // within each): sequence b owns Hkv * q_len * G * S of them when its
  // lengths are valid.  An exclusive scan over the cached lengths (four per
  // thread) gives each sequence's first unit, so the warps share exactly
  // the live units and none takes more than ceil(live / warps).  Without
  // the cache (very large batches) the warps walk every unit of the
  // launch's capacity and skip the dead ones.
  const bool compact = nb_cache > 0 && nunits < 0x7fffffffLL;
  if (compact) {
    int cnt[4], sum = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int b = 4 * tid + k;
      cnt[k] = 0;
      if (b < nb_cache) {
        const Len l{lens[b].x, lens[b].y};
        if (live_row(p, l, 0)) cnt[k] = p.Hkv * l.ql * p.G * S;
      }
      sum += cnt[k];
    }
    int incl = sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += t;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      int w = lane < kWarps ? wsum[lane] : 0;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, w, off);
        if (lane >= off) w += t;
      }
      if (lane < kWarps) wsum[lane] = w;
    }
    __syncthreads();
    int base = (warp > 0 ? wsum[warp - 1] : 0) + incl - sum;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int b = 4 * tid + k;
      if (b < nb_cache) ustart[b] = base;
      base += cnt[k];
    }
    if (tid == 0) ustart[nb_cache] = wsum[kWarps - 1];
  }

  // ---- wait until the split kernel's partials are complete and visible
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  for (int e = tid; e < ntab; e += kCombineThreads) tab[e] = p.plan_tab[e];
  __syncthreads();

  const float kNegInf = -__int_as_float(0x7f800000);
  const int g = lane >> 3, f = lane & 7;
  // units interleaved over the blocks (warp w of block x takes w * grid + x,
  // then steps by the grid's warp count), so every SM gets a share
  const int64_t nwork = compact ? (int64_t)ustart[nb_cache] : nunits;
  const int64_t tw = (int64_t)gridDim.x * kWarps;
  for (int64_t x = (int64_t)warp * gridDim.x + blockIdx.x; x < nwork; x += tw) {
    int s, r, h, b;
    Len l;
    if (compact) {
      const int v = (int)x;
      b = find_seq(ustart, nb_cache, v);
      l = Len{lens[b].x, lens[b].y};
      const int rl = l.ql * p.G;  // live rows of this sequence per KV head
      const int loc = v - ustart[b];
      s = loc % S;
      const int rr = loc / S;
      r = rr % rl;
      h = rr / rl;
    } else {
      // unit -> (b, h, row, slice); slices fastest
      s = (int)(x % S);
      const int64_t ur = x / S;
      r = (int)(ur % R);
      const int64_t bh = ur / R;
      h = (int)(bh % p.Hkv);
      b = (int)(bh / p.Hkv);
      l = len_of(b);
      if (!live_row(p, l, r / p.G)) continue;  // zero-filled above (uniform per warp)
    }
    const int i = r / p.G, gg = r - i * p.G;
    // partitions of this (sequence, KV head): slots slot0 .. slot0 + nP - 1
    int slot0 = 0, nP = 0;
    if (!p.dev_plan) {
      slot0 = (b * p.Hkv + h) * p.P;
      const int T = p.t_from_len ? max(64, plan_t_from_len(l.L, p.P)) : p.T;
      nP = (l.L + T - 1) / T;
    } else {
      const int2 e = b * p.Hkv + h < ntab ? tab[b * p.Hkv + h] : p.plan_tab[b * p.Hkv + h];
      slot0 = e.x;
      nP = e.y;
      if (slot0 < 0 || nP < 1 || nP > p.P || slot0 + nP > p.plan_G) {  // never: a library bug
        if (lane == 0) atomicOr(p.status, VAE4_STATUS_PLAN);
        nP = 0;
      }
    }
    const int64_t pstride = (int64_t)p.rows_pad;  // rows per partition slot
    const float *ml = p.ws_ml + ((int64_t)slot0 * pstride + r) * 2;
    const float *o = p.ws_o + ((int64_t)slot0 * pstride + r) * p.D + 32 * s + 4 * f;
    const int64_t ostride = pstride * p.D;

    // the head's V scale, requested with the partials (not after them)
    const float sv = __ldg(p.scales + h * p.scale_sh + 1);
    float M = kNegInf, lam = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    bool bad = false;
    for (int c0 = 0; c0 < nP; c0 += CH) {
      // this lane's partitions q = c0 + g + PG k: (max, sum) pairs first,
      // then the O partials, all in flight together
      float2 mlr[NPL];
      float4 v[NPL];
#pragma unroll
      for (int k = 0; k < NPL; ++k) {
        const int q = c0 + g + PG * k;
        mlr[k] = q < nP ? __ldcg(reinterpret_cast<const float2 *>(ml + (int64_t)q * pstride * 2))
                        : make_float2(kNegInf, 0.f);
      }
#pragma unroll
      for (int k = 0; k < NPL; ++k) {
        const int q = c0 + g + PG * k;
        v[k] = q < nP ? __ldcg(reinterpret_cast<const float4 *>(o + (int64_t)q * ostride))
                      : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      // maximum over live partitions (l > 0); a negative sum marks a
      // partition that met an invalid page or timed out
      float mx = M;
#pragma unroll
      for (int k = 0; k < NPL; ++k) {
        if (mlr[k].y > 0.f) mx = fmaxf(mx, mlr[k].x);
        bad |= mlr[k].y < 0.f;
      }
#pragma unroll
      for (int off = 8; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      if (mx != M) {  // this chunk raised the maximum: rescale the sums so far
        const float c = M == kNegInf ? 0.f : exp2f(M - mx);
        lam *= c;
        acc.x *= c;
        acc.y *= c;
        acc.z *= c;
        acc.w *= c;
        M = mx;
      }
      // w = 2^(m - M); sums over this lane's partitions in ascending order
#pragma unroll
      for (int k = 0; k < NPL; ++k) {
        const float w = mlr[k].y > 0.f ? (mlr[k].x == M ? 1.f : exp2f(mlr[k].x - M)) : 0.f;
        lam += w * mlr[k].y;
        acc.x += w * v[k].x;
        acc.y += w * v[k].y;
        acc.z += w * v[k].z;
        acc.w += w * v[k].w;
      }
    }
    // the four partition groups of the warp, by a fixed tree (lane bits 3, 4)
#pragma unroll
    for (int off = 8; off < 32; off <<= 1) {
      lam += __shfl_xor_sync(0xffffffffu, lam, off);
      acc.x += __shfl_xor_sync(0xffffffffu, acc.x, off);
      acc.y += __shfl_xor_sync(0xffffffffu, acc.y, off);
      acc.z += __shfl_xor_sync(0xffffffffu, acc.z, off);
      acc.w += __shfl_xor_sync(0xffffffffu, acc.w, off);
    }
    bad = __any_sync(0xffffffffu, bad);
    if (lane < 8) {
      uint2 res = make_uint2(0u, 0u);
      if (!bad && lam > 0.f) {
        const float beta = sv * 256.0f;  // partials hold dec(V) * 2^-8
        const __half2 lo = __floats2half2_rn(__fdiv_rn(acc.x, lam) * beta, __fdiv_rn(acc.y, lam) * beta);
        const __half2 hi = __floats2half2_rn(__fdiv_rn(acc.z, lam) * beta, __fdiv_rn(acc.w, lam) * beta);
        res.x = *reinterpret_cast<const uint32_t *>(&lo);
        res.y = *reinterpret_cast<const uint32_t *>(&hi);
      }
      __half *out = static_cast<__half *>(p.out) + (int64_t)b * p.o_sb + (int64_t)i * p.o_si +
                    (int64_t)(h * p.G + gg) * p.o_sh + 32 * s + 4 * f;
      *reinterpret_cast<uint2 *>(out) = res;
    }
  }
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
  if (p.D % 32 != 0) return cudaErrorInvalidValue;
  if (!p.dev_plan && p.P > 32) {  // one stream over many partitions: a CTA per (row, 64 d)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.Qmax * p.G * (p.D / 64), p.Hkv, p.B);
    cfg.blockDim = dim3(kRowThreads);
    cfg.dynamicSmemBytes = (size_t)p.P * 2 * sizeof(float);  // (m_p, l_p) per partition
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const int smem = (int)cfg.dynamicSmemBytes;
    if (smem > 48 * 1024) {  // beyond the default dynamic shared-memory limit
      const cudaError_t e = cudaFuncSetAttribute(combine_rows_kernel,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (e != cudaSuccess) return e;
    }
    return cudaLaunchKernelEx(&cfg, combine_rows_kernel, p);
  }
  // enough blocks for every unit of the launch's capacity, at most the
  // resident blocks of one wave (units past it: grid-stride loop)
  const int64_t units = (int64_t)p.B * p.Hkv * p.Qmax * p.G * (p.D / 32);
  const int64_t cap = 2 * (p.num_sms > 0 ? p.num_sms : 148);  // two blocks per SM
  int64_t nblk = (units + kWarps - 1) / kWarps;
  nblk = nblk < 1 ? 1 : (nblk > cap ? cap : nblk);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)nblk, 1, 1);
  cfg.blockDim = dim3(kCombineThreads);
  const int nb_cache = p.B <= kCacheB ? p.B : 0;
  const int ntab = (p.dev_plan && p.B * p.Hkv <= kCacheTab) ? p.B * p.Hkv : 0;
  // lengths, stream table, first live unit per sequence
  cfg.dynamicSmemBytes = (size_t)(nb_cache + ntab) * sizeof(int2) +
                         (size_t)(nb_cache + 1) * sizeof(int);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, combine_kernel, p);
}

cudaError_t launch_decode_table(uint16_t *out, bool integer_path, bool e5m2,
                                cudaStream_t stream) {
  decode_table_kernel<<<1, 64, 0, stream>>>(out, integer_path, e5m2);
  return cudaGetLastError();
}

}  // namespace vae4
