// Streaming-read reference kernel for the roofline: reads every KV byte that
// the verify step with the same arguments reads -- for each (sequence b, KV
// head h) the K and V slices of tokens 0 .. L-1, gathered through the block
// table in the same page order -- with plain 16-byte loads and no compute.
// Its time is the practical floor of the step's page gather on this GPU, the
// number the step's own time is compared with.
//
// Work unit = one (b, h, logical page): its K and V slices (page * D bytes
// each, fewer for the last, partial page) are read by one warp, 16 bytes per
// lane per load, K and V loads interleaved, up to 16 loads in flight per
// lane.  The loaded 32-bit words are XOR-folded into the word at workspace
// byte 128 (inside the status block, away from the status word), so the
// loads cannot be removed and a caller that zeroes that word first reads back
// the XOR of every word the step reads.  Invalid lengths or page ids are
// skipped (the verify step reports them; this kernel only measures).
#include "common.cuh"
#include "kernels.h"

namespace vae4 {

namespace {

constexpr int kReadThreads = 512;

template <int CH>  // 16-byte chunks per lane per batch (<= 8)
__global__ void __launch_bounds__(kReadThreads) kv_read_kernel(const SplitParams p) {
  const int warps = gridDim.x * (kReadThreads / 32);
  const int w = blockIdx.x * (kReadThreads / 32) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  const int64_t slice = (int64_t)p.page * p.D;  // bytes of one K or V page slice
  uint32_t acc = 0;
  for (int b = 0; b < p.B; ++b) {
    const int L = p.seq[(int64_t)b * p.seq_sb];
    if (L <= 0 || L > p.capacity) continue;
    const int npg = (L + p.page - 1) / p.page;
    const int units = npg * p.Hkv;
    for (int u = w; u < units; u += warps) {
      const int lp = u / p.Hkv, h = u - lp * p.Hkv;
      const int phys = p.bt[(int64_t)b * p.bt_sb + lp];
      if (phys < 0 || phys >= p.n_pages) continue;
      const int toks = min(p.page, L - lp * p.page);
      const int64_t valid = (int64_t)toks * p.D;  // bytes of this slice that are read
      const uint8_t *k = p.kv + ((int64_t)phys * 2 * p.Hkv + h) * slice;
      const uint8_t *v = k + (int64_t)p.Hkv * slice;
      for (int64_t base = 0; base < valid; base += CH * 512) {
        uint4 rk[CH], rv[CH];
#pragma unroll
        for (int c = 0; c < CH; ++c) {
          const int64_t off = base + (int64_t)(c * 32 + lane) * 16;
          const bool ok = off < valid;
          rk[c] = ok ? __ldcs(reinterpret_cast<const uint4 *>(k + off)) : make_uint4(0, 0, 0, 0);
          rv[c] = ok ? __ldcs(reinterpret_cast<const uint4 *>(v + off)) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int c = 0; c < CH; ++c)
          acc ^= rk[c].x ^ rk[c].y ^ rk[c].z ^ rk[c].w ^ rv[c].x ^ rv[c].y ^ rv[c].z ^ rv[c].w;
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc ^= __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0 && acc != 0u) atomicXor(p.status + 32, acc);
}

}  // namespace

cudaError_t launch_kv_read(const SplitParams &p, int num_sms, cudaStream_t stream) {
  const int64_t slice = (int64_t)p.page * p.D;
  if (slice % 512 != 0) return cudaErrorInvalidValue;
  const int grid = 4 * (num_sms > 0 ? num_sms : 1);
  switch (slice / 512) {
    case 2: kv_read_kernel<2><<<grid, kReadThreads, 0, stream>>>(p); break;  // page 16, D 64
    case 4: kv_read_kernel<4><<<grid, kReadThreads, 0, stream>>>(p); break;  // 16 x 128, 32 x 64
    default: kv_read_kernel<8><<<grid, kReadThreads, 0, stream>>>(p); break; // 8 KB+ per slice
  }
  return cudaGetLastError();
}

}  // namespace vae4
