// Split (partition) kernel on the warp-level tensor-core path (mma.sync
// m16n8k16, FP16 operands, FP32 accumulate).
//
// One CTA = one (partition p, KV head h, sequence b).  It streams the E4M3
// K/V bytes of its token range through a 3-stage cp.async ring (16-byte
// copies straight from the block-table pages), decodes them exactly to FP16
// in shared memory, and runs Q.K^T, a masked online softmax and P.V on the
// tensor cores with the rows (query x group head) as the MMA M dimension.
// The running max, running sum and unnormalised P.V stay FP32 and are
// written to the workspace for the combine kernel, which alone merges them
// (PR #524 "[Kernel][SM70] Add opt-in E4M3 grouped attention with FP32
// partials", final status).  Keys are consumed in ascending logical order,
// the order the audited kernel fixes for its partitions and its P.V sums
// (PR #566, Purpose and Final audit), so the result depends only on logical
// token positions: moving pages changes no bit.
#include "common.cuh"
#include "kernels.h"
#include "plan.cuh"
#include "verify_attn_e4m3.h"

namespace vae4 {

namespace {

constexpr int kTK = 64;     // keys per tile (4 pages of 16 tokens)
constexpr int kStages = 3;  // depth of the raw-byte ring

// Byte offset of 16-byte chunk c of row r in a [rows][D] FP16 tile whose
// rows are D*2 bytes; chunks are XOR-swizzled by row so ldmatrix reads of 8
// consecutive rows hit 8 distinct bank groups.
template <int D>
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return static_cast<uint32_t>(r * (D * 2) + ((c ^ (r & 7)) << 4));
}

template <int D>
__global__ void __launch_bounds__(192, 1) split_mma_kernel(const SplitParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int ROWB = D * 2;      // bytes per FP16 row
  constexpr int QCH = D / 8;       // 16-byte chunks per FP16 row
  constexpr int CH = D / 16;       // 16-byte chunks per E4M3 row
  constexpr int RAW = kTK * D;     // raw bytes of K (or V) per tile
  constexpr int NT = D / 8;        // n-tiles of the output
  constexpr float kLog2e = 1.4426950408889634f;
  const float kInf = __int_as_float(0x7f800000);

  uint8_t *Qs = smem;
  uint8_t *Ks = Qs + p.rows_pad * ROWB;
  uint8_t *Vs = Ks + kTK * ROWB;
  uint8_t *raw = Vs + kTK * ROWB;

  const int tid = threadIdx.x, nthr = blockDim.x;
  const int warp = tid >> 5, lane = tid & 31;
  // static grid (partition, head, sequence) or the device-side balanced
  // plan (grid.x = partition number), evaluated by every warp
  int part, h, b, T;
  int64_t pslot;
  if (p.dev_plan) {
    const PlanIn in{p.seq, p.seq_sb, p.seq_has_qlen, p.Qmax, p.capacity, p.B, p.Hkv, p.plan_G,
                    p.G, p.plan_N};
    const PlanCta c = plan_cta_global(in, blockIdx.x, lane);
    if (c.p < 0) return;  // past the plan
    b = c.b;
    h = c.h;
    part = c.p;
    T = c.W;
    pslot = blockIdx.x;
    if (part == 0 && tid == 0) p.plan_tab[b * p.Hkv + h] = make_int2((int)blockIdx.x, c.np);
  } else {
    part = blockIdx.x;
    h = blockIdx.y;
    b = blockIdx.z;
    T = p.T;
    pslot = (int64_t)(b * p.Hkv + h) * p.P + part;
  }

  const int L = p.seq[(int64_t)b * p.seq_sb];
  const int ql = p.seq_has_qlen ? p.seq[(int64_t)b * p.seq_sb + 1] : p.Qmax;
  if (L < 0 || L > p.capacity) {
    if (part == 0 && h == 0 && tid == 0) atomicOr(p.status, VAE4_STATUS_BAD_LENGTH);
    return;
  }
  if (ql < 0 || ql > p.Qmax || (L > 0 && ql > L)) {
    if (part == 0 && h == 0 && tid == 0) atomicOr(p.status, VAE4_STATUS_BAD_QLEN);
    return;
  }
  if (!p.dev_plan && p.t_from_len && L > 0) T = max(64, plan_t_from_len(L, p.P));
  const int k0 = part * T;
  if (k0 >= L) return;  // dead partition: never read by the combine
  const int k1 = min(k0 + T, L);
  const int ntiles = (k1 - k0 + kTK - 1) / kTK;

  // ---- queries: rows r = i*G + g of this KV head, padding rows zeroed
  const __half *qb = static_cast<const __half *>(p.q) + (int64_t)b * p.q_sb;
  for (int c = tid; c < p.rows_pad * QCH; c += nthr) {
    const int r = c / QCH, cc = c - r * QCH;
    const int i = r / p.G, g = r - i * p.G;
    const bool ok = r < p.rows && i < ql;
    const __half *src = ok ? qb + i * p.q_si + (int64_t)(h * p.G + g) * p.q_sh + cc * 8 : qb;
    cp_async16(smem_u32(Qs + swz<D>(r, cc)), src, ok);
  }
  cp_async_commit();

  // ---- raw K/V tile issue: 16-byte copies from the block-table pages
  bool bad_block = false;
  auto issue = [&](int t, int stage) {
    const int kt = k0 + t * kTK;
    uint8_t *rs = raw + stage * 2 * RAW;
    for (int c = tid; c < 2 * kTK * CH; c += nthr) {
      const int sel = c / (kTK * CH);
      const int rem = c - sel * (kTK * CH);
      const int kl = rem / CH, dc = rem - kl * CH;
      const int key = kt + kl;
      bool ok = key < k1;
      const uint8_t *src = p.kv;
      if (ok) {
        const int lp = key / p.page;
        const int phys = p.bt[(int64_t)b * p.bt_sb + lp];
        if (phys < 0 || phys >= p.n_pages) {
          bad_block = true;
          ok = false;
        } else {
          src = p.kv + ((((int64_t)phys * 2 + sel) * p.Hkv + h) * p.page + (key - lp * p.page)) * D +
                dc * 16;
        }
      }
      cp_async16(smem_u32(rs + sel * RAW + kl * D + dc * 16), src, ok);
    }
  };

  // ---- per-warp state: warp w owns rows 16w .. 16w+15
  const int mw = p.rows_pad >> 4;
  const bool mma_warp = warp < mw;
  const int r0 = warp * 16 + (lane >> 2), r1 = r0 + 8;
  auto last_key = [&](int r) {
    const int i = r / p.G;
    return (r < p.rows && i < ql) ? L - ql + i : -1;
  };
  const int pos0 = last_key(r0), pos1 = last_key(r1);
  // K holds dec*2^-8, so the score is S * 2^8 * s_K * sm_scale; work in log2
  const float alpha = p.sm_scale * p.scales[h * p.scale_sh] * 256.0f * kLog2e;

  float oacc[NT][4];
#pragma unroll
  for (int n = 0; n < NT; ++n) oacc[n][0] = oacc[n][1] = oacc[n][2] = oacc[n][3] = 0.f;
  float m_run0 = -kInf, m_run1 = -kInf, l_run0 = 0.f, l_run1 = 0.f;

#pragma unroll
  for (int s = 0; s < kStages - 1; ++s) {
    if (s < ntiles) issue(s, s);
    cp_async_commit();
  }

  for (int t = 0; t < ntiles; ++t) {
    if (t + kStages - 1 < ntiles) issue(t + kStages - 1, (t + kStages - 1) % kStages);
    cp_async_commit();
    cp_async_wait<kStages - 1>();
    __syncthreads();

    // ---- exact decode of the raw stage into the FP16 K/V tiles
    const uint8_t *rs = raw + (t % kStages) * 2 * RAW;
    for (int c = tid; c < 2 * kTK * CH; c += nthr) {
      const int sel = c / (kTK * CH);
      const int rem = c - sel * (kTK * CH);
      const int kl = rem / CH, dc = rem - kl * CH;
      const uint4 w = *reinterpret_cast<const uint4 *>(rs + sel * RAW + kl * D + dc * 16);
      uint4 h0, h1;
      e4m3x16_to_f16x16(w, h0, h1);
      uint8_t *dst = sel ? Vs : Ks;
      *reinterpret_cast<uint4 *>(dst + swz<D>(kl, 2 * dc)) = h0;
      *reinterpret_cast<uint4 *>(dst + swz<D>(kl, 2 * dc + 1)) = h1;
    }
    __syncthreads();

    if (mma_warp) {
      // ---- S = Q K^T for 16 rows x 64 keys
      float sacc[8][4];
#pragma unroll
      for (int n = 0; n < 8; ++n) sacc[n][0] = sacc[n][1] = sacc[n][2] = sacc[n][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        uint32_t a[4];
        ldsm_x4(a, smem_u32(Qs + swz<D>(warp * 16 + (lane & 15), 2 * ks + (lane >> 4))));
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t bb[4];
          ldsm_x4(bb, smem_u32(Ks + swz<D>(16 * c + ((lane >> 4) & 1) * 8 + (lane & 7),
                                           2 * ks + ((lane >> 3) & 1))));
          mma16816(sacc[2 * c], a, bb[0], bb[1]);
          mma16816(sacc[2 * c + 1], a, bb[2], bb[3]);
        }
      }

      // ---- causal/partition mask, online softmax in FP32 (log2 domain)
      const int kt = k0 + t * kTK;
      float mx0 = -kInf, mx1 = -kInf;
#pragma unroll
      for (int n = 0; n < 8; ++n) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int key = kt + 8 * n + 2 * (lane & 3) + (e & 1);
          const int pos = e < 2 ? pos0 : pos1;
          const float x = (key <= pos && key < k1) ? sacc[n][e] * alpha : -kInf;
          sacc[n][e] = x;
          if (e < 2) mx0 = fmaxf(mx0, x); else mx1 = fmaxf(mx1, x);
        }
      }
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      const float mn0 = fmaxf(m_run0, mx0), mn1 = fmaxf(m_run1, mx1);
      const float base0 = mn0 == -kInf ? 0.f : mn0;
      const float base1 = mn1 == -kInf ? 0.f : mn1;
      const float c0 = m_run0 == mn0 ? 1.f : fast_exp2(m_run0 - base0);
      const float c1 = m_run1 == mn1 ? 1.f : fast_exp2(m_run1 - base1);
      m_run0 = mn0;
      m_run1 = mn1;
      uint32_t pa[8][2];
      float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
      for (int n = 0; n < 8; ++n) {
        const __half2 h01 = __floats2half2_rn(fast_exp2(sacc[n][0] - base0),
                                              fast_exp2(sacc[n][1] - base0));
        const __half2 h23 = __floats2half2_rn(fast_exp2(sacc[n][2] - base1),
                                              fast_exp2(sacc[n][3] - base1));
        // the running sum adds the same FP16-rounded p that enters P.V
        const float2 f01 = __half22float2(h01), f23 = __half22float2(h23);
        ls0 += f01.x + f01.y;
        ls1 += f23.x + f23.y;
        pa[n][0] = *reinterpret_cast<const uint32_t *>(&h01);
        pa[n][1] = *reinterpret_cast<const uint32_t *>(&h23);
      }
      l_run0 = l_run0 * c0 + ls0;
      l_run1 = l_run1 * c1 + ls1;
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        oacc[n][0] *= c0;
        oacc[n][1] *= c0;
        oacc[n][2] *= c1;
        oacc[n][3] *= c1;
      }

      // ---- O += P V
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint32_t a[4] = {pa[2 * kk][0], pa[2 * kk][1], pa[2 * kk + 1][0], pa[2 * kk + 1][1]};
#pragma unroll
        for (int np = 0; np < D / 16; ++np) {
          uint32_t bb[4];
          ldsm_x4_t(bb, smem_u32(Vs + swz<D>(16 * kk + ((lane >> 3) & 1) * 8 + (lane & 7),
                                             2 * np + (lane >> 4))));
          mma16816(oacc[2 * np], a, bb[0], bb[1]);
          mma16816(oacc[2 * np + 1], a, bb[2], bb[3]);
        }
      }
    }
    __syncthreads();  // the next decode overwrites Ks/Vs
  }
  cp_async_wait<0>();

  const bool bad = __syncthreads_or(bad_block);
  if (bad && tid == 0) atomicOr(p.status, VAE4_STATUS_BAD_BLOCK);

  if (mma_warp) {
    l_run0 += __shfl_xor_sync(0xffffffffu, l_run0, 1);
    l_run0 += __shfl_xor_sync(0xffffffffu, l_run0, 2);
    l_run1 += __shfl_xor_sync(0xffffffffu, l_run1, 1);
    l_run1 += __shfl_xor_sync(0xffffffffu, l_run1, 2);
    const int64_t slot = pslot * p.rows_pad;
    if ((lane & 3) == 0) {
      p.ws_ml[(slot + r0) * 2 + 0] = m_run0;
      p.ws_ml[(slot + r0) * 2 + 1] = bad ? -1.f : l_run0;
      p.ws_ml[(slot + r1) * 2 + 0] = m_run1;
      p.ws_ml[(slot + r1) * 2 + 1] = bad ? -1.f : l_run1;
    }
    float *o0 = p.ws_o + (slot + r0) * D + 2 * (lane & 3);
    float *o1 = p.ws_o + (slot + r1) * D + 2 * (lane & 3);
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      *reinterpret_cast<float2 *>(o0 + 8 * n) = make_float2(oacc[n][0], oacc[n][1]);
      *reinterpret_cast<float2 *>(o1 + 8 * n) = make_float2(oacc[n][2], oacc[n][3]);
    }
  }
}

}  // namespace

size_t split_mma_smem_bytes(int D, int rows_pad) {
  return (size_t)rows_pad * D * 2 + 2 * (size_t)kTK * D * 2 + (size_t)kStages * 2 * kTK * D;
}

int split_mma_threads(int rows_pad) {
  const int mw = rows_pad / 16;
  return 32 * (mw < 4 ? 4 : mw);
}

cudaError_t launch_split_mma(const SplitParams &p, cudaStream_t stream) {
  const size_t smem = split_mma_smem_bytes(p.D, p.rows_pad);
  const dim3 grid = p.dev_plan ? dim3(p.plan_G, 1, 1) : dim3(p.P, p.Hkv, p.B);
  const dim3 block(split_mma_threads(p.rows_pad));
  cudaError_t e = cudaSuccess;
  switch (p.D) {
    case 64:
      e = cudaFuncSetAttribute(split_mma_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e == cudaSuccess) split_mma_kernel<64><<<grid, block, smem, stream>>>(p);
      break;
    case 128:
      e = cudaFuncSetAttribute(split_mma_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e == cudaSuccess) split_mma_kernel<128><<<grid, block, smem, stream>>>(p);
      break;
    case 256:
      e = cudaFuncSetAttribute(split_mma_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e == cudaSuccess) split_mma_kernel<256><<<grid, block, smem, stream>>>(p);
      break;
    default:
      return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace vae4
