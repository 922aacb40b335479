// C-ABI entry points: argument validation, the split-K partition plan, the
// workspace layout and the kernel launches.  See include/verify_attn_e4m3.h
// for the contract of every function.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <cmath>

#include "kernels.h"
#include "params.h"
#include "verify_attn_e4m3.h"

namespace {

using vae4::CombineParams;
using vae4::kDevPlanMaxB;
using vae4::SplitParams;

constexpr int64_t kStatusBytes = 256;  // status word + padding
constexpr int kMaxRowsPad = 96;        // Qmax * G rounded to 16 (q16 x GQA6)
constexpr int kMaxQmax = 16;
constexpr int64_t kMaxPartitions = 8192;  // per (sequence, KV head)

int64_t align_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

// Rows of FP32 partial state per (sequence, KV head, partition): enough for
// both split kernels' row layouts.
int64_t ws_rows(int rows) {
  int n_rg = 1, n = 16;
  vae4::tc_row_groups(rows, &n_rg, &n);
  return std::max<int64_t>(align_up(rows, 16), (int64_t)n_rg * n);
}

struct WsLayout {
  int64_t ml_off, o_off, tab_off, total;
};

// status | (max, sum) [slots][rows][2] | unnormalised O [slots][rows][D] |
// (first slot, partitions) [B][Hkv] of the device-side plan
WsLayout ws_layout(int64_t slots, int rows_pad, int D, int64_t streams) {
  WsLayout l;
  l.ml_off = kStatusBytes;
  const int64_t ml_bytes = slots * rows_pad * 2 * 4;
  l.o_off = align_up(l.ml_off + ml_bytes, 256);
  l.tab_off = align_up(l.o_off + slots * rows_pad * D * 4, 256);
  l.total = l.tab_off + streams * 8;  // device plan: (first slot, partitions) per stream
  return l;
}

// CTAs of the device-side plan: one wave on the SMs, at least one CTA per
// (sequence, KV head, row group) so one partition per stream always fits.
int vae4_tc_groups(int rows) {  // row groups of the tcgen05 kernel (the most any path uses)
  int g = 1, n = 16;
  vae4::tc_row_groups(rows, &g, &n);
  return g;
}

int64_t dev_plan_ctas(int B, int Hkv, int n_rg, int sms) {
  return std::max<int64_t>(sms, (int64_t)B * Hkv * n_rg);
}

// Partial slots a launch needs: the static plan's B * Hkv * P, or with an
// automatic plan of a batch the device plan's grid, whichever is larger.
int64_t ws_slots(int B, int Hkv, int P, int T_req, int sms, int n_rg) {
  int64_t s = (int64_t)B * Hkv * P;
  if (T_req == 0 && B > 1 && B <= kDevPlanMaxB && (int64_t)B * Hkv * n_rg <= 65535)
    s = std::max<int64_t>(s, dev_plan_ctas(B, Hkv, n_rg, sms));
  return s;
}

// The device-side plan's partition length when every one of the B
// sequences has L = cap and r row groups (the same steps as the device
// code, with the counts in closed form): the guess the split kernel
// prefetches block-table entries for while it reads the actual lengths.
int plan_width_equal(int B, int Hkv, int G, int cap, int r) {
  const int64_t gb = G / Hkv, nrg = (int64_t)B * r, sum = nrg * cap;
  auto up16 = [](int64_t x) { return (int)std::min<int64_t>((x + 15) & ~(int64_t)15, 0x7FFFFFF0); };
  auto count = [&](int W) { return nrg * ((cap + W - 1) / W); };
  int lo = std::max(64, up16((sum + gb - 1) / gb));
  if (count(lo) <= gb) return lo;
  int hi = std::max(64, up16(cap));
  if (gb > nrg && sum / 65536 / (gb - nrg) < (1 << 14))
    hi = std::min(hi, up16((sum + (gb - nrg) - 1) / (gb - nrg)));
  hi = std::max(hi, lo);
  for (int it = 0; it < 6 && hi - lo > 16; ++it) {
    const int mid = (int)(((int64_t)lo + hi) / 32 * 16);
    if (count(mid) <= gb)
      hi = mid;
    else
      lo = mid;
  }
  return hi;
}

int do_plan(int B, int Hkv, int cap, int T_req, int num_sms, int *T_out, int *P_out) {
  if (B < 1 || Hkv < 1 || cap < 1 || num_sms < 1) return VAE4_ERR_SHAPE;
  int64_t T;
  if (T_req < 0 || (T_req > 0 && T_req % 16 != 0)) return VAE4_ERR_PARTITION;
  if (T_req > 0) {
    T = T_req;
  } else {
    const int64_t units = (int64_t)B * Hkv;
    const int64_t pmax = std::max<int64_t>(1, num_sms / units);
    T = align_up((cap + pmax - 1) / pmax, 16);
    T = std::max<int64_t>(T, 64);
  }
  const int64_t P = (cap + T - 1) / T;
  if (P > kMaxPartitions) return VAE4_ERR_PARTITION;
  *T_out = (int)T;
  *P_out = (int)P;
  return VAE4_OK;
}

int device_sms(int *out) {
  static int cache[128] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return VAE4_ERR_CUDA;
  if (dev >= 0 && dev < 128 && cache[dev] > 0) {
    *out = cache[dev];
    return VAE4_OK;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
    return VAE4_ERR_CUDA;
  if (dev >= 0 && dev < 128) cache[dev] = n;
  *out = n;
  return VAE4_OK;
}

bool al16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// q / out: F16 [B][Qmax][Hq][D], stride[3] == 1, other strides multiples of 8.
int check_qo(const vae4_tensor *t) {
  if (t->dtype != VAE4_F16) return VAE4_ERR_DTYPE;
  if (t->ndim != 4) return VAE4_ERR_SHAPE;
  for (int k = 0; k < 4; ++k)
    if (t->shape[k] < 0) return VAE4_ERR_SHAPE;
  if (t->stride[3] != 1) return VAE4_ERR_STRIDE;
  for (int k = 0; k < 3; ++k)
    if (t->stride[k] % 8 != 0 || t->stride[k] < 0) return VAE4_ERR_STRIDE;
  if (!al16(t->data)) return VAE4_ERR_MISALIGNED;
  return VAE4_OK;
}

// A validated KV cache: the pool form (one tensor, the mma.sync kernel and
// the gather floor read it too) or separate K and V caches with strides.
struct KvSrc {
  const uint8_t *pool;  // pool form, else null
  const uint8_t *kb, *vb;
  int64_t k_ps, k_ts, k_hs, v_ps, v_ts, v_hs;  // bytes
  int64_t n_pages, Hkv, page;
};

// kv pages: U8 [n_pages][2][Hkv][page][D], contiguous
int check_pool(const vae4_tensor *kv, int64_t D, KvSrc *o) {
  if (kv->dtype != VAE4_U8) return VAE4_ERR_DTYPE;
  if (kv->ndim != 5 || kv->shape[1] != 2 || kv->shape[4] != D || kv->shape[0] < 1 ||
      kv->shape[2] < 1)
    return VAE4_ERR_SHAPE;
  const int64_t n_pages = kv->shape[0], Hkv = kv->shape[2], page = kv->shape[3];
  // any multiple of 16 tokens: the kernels move 16-key page slices
  if (page < 16 || page % 16 != 0 || page > 65536) return VAE4_ERR_UNSUPPORTED;
  if (kv->stride[4] != 1 || kv->stride[3] != D || kv->stride[2] != page * D ||
      kv->stride[1] != Hkv * page * D || kv->stride[0] != 2 * Hkv * page * D)
    return VAE4_ERR_STRIDE;
  if (!al16(kv->data)) return VAE4_ERR_MISALIGNED;
  if (n_pages * 2 * Hkv * page > (int64_t)0x7fffff00) return VAE4_ERR_SHAPE;
  const uint8_t *b = static_cast<const uint8_t *>(kv->data);
  o->pool = b;
  o->kb = b;
  o->vb = b ? b + Hkv * page * D : nullptr;
  o->k_ps = o->v_ps = 2 * Hkv * page * D;
  o->k_ts = o->v_ts = D;
  o->k_hs = o->v_hs = page * D;
  o->n_pages = n_pages;
  o->Hkv = Hkv;
  o->page = page;
  return VAE4_OK;
}

// separate caches: U8 [n_pages][page][Hkv][D] each, same shape, d
// contiguous, other strides any multiples of 8 bytes, bases 8-byte aligned
int check_kv(const vae4_tensor *k, const vae4_tensor *v, int64_t D, KvSrc *o) {
  for (const vae4_tensor *t : {k, v}) {
    if (t->dtype != VAE4_U8) return VAE4_ERR_DTYPE;
    if (t->ndim != 4 || t->shape[3] != D || t->shape[0] < 1 || t->shape[2] < 1)
      return VAE4_ERR_SHAPE;
    for (int d = 0; d < 4; ++d)
      if (t->shape[d] != k->shape[d]) return VAE4_ERR_SHAPE;
    if (t->stride[3] != 1) return VAE4_ERR_STRIDE;
    for (int d = 0; d < 3; ++d)
      if (t->stride[d] < 0 || t->stride[d] % 8 != 0 || t->stride[d] >= ((int64_t)1 << 40))
        return VAE4_ERR_STRIDE;
    if ((reinterpret_cast<uintptr_t>(t->data) & 7u) != 0) return VAE4_ERR_MISALIGNED;
  }
  const int64_t page = k->shape[1];
  if (page < 16 || page % 16 != 0 || page > 65536) return VAE4_ERR_UNSUPPORTED;
  if (k->shape[0] > 0x7fffffff) return VAE4_ERR_SHAPE;
  o->pool = nullptr;
  o->kb = static_cast<const uint8_t *>(k->data);
  o->vb = static_cast<const uint8_t *>(v->data);
  o->k_ps = k->stride[0];
  o->k_ts = k->stride[1];
  o->k_hs = k->stride[2];
  o->v_ps = v->stride[0];
  o->v_ts = v->stride[1];
  o->v_hs = v->stride[2];
  o->n_pages = k->shape[0];
  o->Hkv = k->shape[2];
  o->page = page;
  return VAE4_OK;
}

struct Prepared {
  SplitParams sp;
  CombineParams cp;
  int64_t ws_needed;
  bool empty;
  bool warp_mma;
  int num_sms;
  long long wait_limit;
};

// SM cycles a pipeline wait of the tcgen05 kernel may take before the CTA
// gives up (about a second at the GB300 clock).
constexpr long long kWaitLimitCycles = 2000000000LL;
// VAE4_FLAG_TEST_SHORT_WAITS: every pipeline wait gives up after this many
// cycles, far less than a memory round trip, so the call takes the abort path
constexpr long long kShortWaitCycles = 256;

cudaError_t launch_split(const Prepared &pr, cudaStream_t st) {
  return pr.warp_mma ? vae4::launch_split_mma(pr.sp, st)
                     : vae4::launch_split_tc(pr.sp, pr.wait_limit, st);
}

// kv: the pool; or k and v (kv == null): separate caches
int prepare(const vae4_tensor *q, const vae4_tensor *kv, const vae4_tensor *kc,
            const vae4_tensor *vc, const vae4_tensor *bt, const vae4_tensor *seq,
            const vae4_tensor *sc, const vae4_tensor *out, const vae4_tensor *ws,
            const vae4_options *opt, Prepared *pr) {
  if (!q || !(kv || (kc && vc)) || !bt || !seq || !sc || !out || !ws) return VAE4_ERR_NULL;
  vae4_options o;
  memset(&o, 0, sizeof(o));
  if (opt) o = *opt;
  if ((o.flags & ~(VAE4_FLAG_WARP_MMA | VAE4_FLAG_KV_E5M2 | VAE4_FLAG_TEST_SHORT_WAITS)) != 0)
    return VAE4_ERR_OPTIONS;
  if (o.hilo_pv != 0 && o.hilo_pv != 1) return VAE4_ERR_OPTIONS;
  if ((o.flags & VAE4_FLAG_WARP_MMA) &&
      ((o.flags & (VAE4_FLAG_KV_E5M2 | VAE4_FLAG_TEST_SHORT_WAITS)) || o.hilo_pv || !kv))
    return VAE4_ERR_UNSUPPORTED;

  int rc = check_qo(q);
  if (rc) return rc;
  rc = check_qo(out);
  if (rc) return rc;
  for (int k = 0; k < 4; ++k)
    if (out->shape[k] != q->shape[k]) return VAE4_ERR_SHAPE;
  const int64_t B = q->shape[0], Qmax = q->shape[1], Hq = q->shape[2], D = q->shape[3];
  if (D != 64 && D != 128 && D != 256) return VAE4_ERR_UNSUPPORTED;
  if (Qmax < 1 || Qmax > kMaxQmax || Hq < 1 || B > 65535) return VAE4_ERR_SHAPE;

  KvSrc src;
  rc = kv ? check_pool(kv, D, &src) : check_kv(kc, vc, D, &src);
  if (rc) return rc;
  const int64_t n_pages = src.n_pages, Hkv = src.Hkv, page = src.page;
  if (Hq % Hkv != 0) return VAE4_ERR_GQA;
  const int64_t G = Hq / Hkv;
  const int64_t rows = Qmax * G;
  if (align_up(rows, 16) > kMaxRowsPad) return VAE4_ERR_UNSUPPORTED;
  const int64_t rows_pad = ws_rows((int)rows);

  // block table: I32 [B][max_pages]
  if (bt->dtype != VAE4_I32) return VAE4_ERR_DTYPE;
  if (bt->ndim != 2 || bt->shape[0] != B || bt->shape[1] < 1) return VAE4_ERR_SHAPE;
  if (bt->stride[1] != 1 || bt->stride[0] < 0) return VAE4_ERR_STRIDE;
  const int64_t max_pages = bt->shape[1];

  // lengths: I32 [B] or [B][2]
  if (seq->dtype != VAE4_I32) return VAE4_ERR_DTYPE;
  int has_qlen = 0;
  if (seq->ndim == 1) {
    if (seq->shape[0] != B) return VAE4_ERR_SHAPE;
  } else if (seq->ndim == 2) {
    if (seq->shape[0] != B || seq->shape[1] != 2) return VAE4_ERR_SHAPE;
    if (seq->stride[1] != 1) return VAE4_ERR_STRIDE;
    has_qlen = 1;
  } else {
    return VAE4_ERR_SHAPE;
  }
  if (seq->stride[0] < 0 || seq->stride[0] > INT32_MAX) return VAE4_ERR_STRIDE;

  // scales: F32 [Hkv][2]
  if (sc->dtype != VAE4_F32) return VAE4_ERR_DTYPE;
  if (sc->ndim != 2 || sc->shape[0] != Hkv || sc->shape[1] != 2) return VAE4_ERR_SHAPE;
  if (sc->stride[1] != 1 || sc->stride[0] < 0 || sc->stride[0] > INT32_MAX) return VAE4_ERR_STRIDE;

  // workspace: U8 [bytes], 256-byte aligned
  if (ws->dtype != VAE4_U8) return VAE4_ERR_DTYPE;
  if (ws->ndim != 1 || ws->stride[0] != 1) return VAE4_ERR_SHAPE;
  if ((reinterpret_cast<uintptr_t>(ws->data) & 255u) != 0) return VAE4_ERR_WORKSPACE;

  const int64_t table_cap = max_pages * page;
  int64_t cap = o.max_seq_len > 0 ? o.max_seq_len : table_cap;
  if (o.max_seq_len < 0 || cap > table_cap || cap > INT32_MAX / 2) return VAE4_ERR_SHAPE;

  int sms = o.num_sms;
  if (sms < 0) return VAE4_ERR_SHAPE;
  if (sms == 0 && B > 0) {
    rc = device_sms(&sms);
    if (rc) return rc;
  }
  int T = 0, P = 0;
  if (B > 0) {
    rc = do_plan((int)B, (int)Hkv, (int)cap, o.partition_tokens, sms, &T, &P);
    if (rc) return rc;
  }
  // automatic plans: one sequence takes its partition length from its L on
  // the device (static grid); a batch gets the device-side balanced plan
  const bool dev_plan = B > 1 && o.partition_tokens == 0 && B <= kDevPlanMaxB &&
                        B * Hkv * vae4_tc_groups((int)rows) <= 65535;
  const bool t_from_len = o.partition_tokens == 0 && !dev_plan;
  // rows per CTA: row groups of the tcgen05 kernel, all rows on the mma.sync path
  int n_rg = 1, n_rows = (int)rows_pad;
  if (!(o.flags & VAE4_FLAG_WARP_MMA)) vae4::tc_row_groups((int)rows, &n_rg, &n_rows);
  const int Gp = (int)dev_plan_ctas((int)B, (int)Hkv, n_rg, sms);  // device plan CTAs
  const WsLayout lay = ws_layout(ws_slots((int)B, (int)Hkv, P, o.partition_tokens, sms,
                                          vae4_tc_groups((int)rows)),
                                 (int)rows_pad, (int)D, B * Hkv);
  pr->ws_needed = lay.total;
  pr->empty = (B == 0);
  pr->warp_mma = (o.flags & VAE4_FLAG_WARP_MMA) != 0;
  pr->wait_limit = (o.flags & VAE4_FLAG_TEST_SHORT_WAITS) ? kShortWaitCycles : kWaitLimitCycles;
  pr->num_sms = sms;
  if (B > 0 && ws->shape[0] < lay.total) return VAE4_ERR_WORKSPACE;
  if (!q->data || !src.kb || !src.vb || !bt->data || !seq->data || !sc->data || !out->data ||
      !ws->data) {
    if (B > 0) return VAE4_ERR_NULL;
  }

  float sm_scale = o.softmax_scale;
  if (!(sm_scale > 0.f)) {
    if (sm_scale != 0.f) return VAE4_ERR_OPTIONS;
    sm_scale = 1.0f / sqrtf((float)D);
  }
  uint8_t *wsb = static_cast<uint8_t *>(ws->data);

  SplitParams &s = pr->sp;
  memset(&s, 0, sizeof(s));
  s.q = q->data;
  s.q_sb = q->stride[0];
  s.q_si = q->stride[1];
  s.q_sh = q->stride[2];
  s.kv = src.pool;
  s.n_pages = n_pages;
  s.k_base = src.kb;
  s.v_base = src.vb;
  s.k_ps = src.k_ps;
  s.k_ts = src.k_ts;
  s.k_hs = src.k_hs;
  s.v_ps = src.v_ps;
  s.v_ts = src.v_ts;
  s.v_hs = src.v_hs;
  s.bt = static_cast<const int32_t *>(bt->data);
  s.bt_sb = bt->stride[0];
  s.max_pages = (int32_t)max_pages;
  s.seq = static_cast<const int32_t *>(seq->data);
  s.seq_sb = (int32_t)seq->stride[0];
  s.seq_has_qlen = has_qlen;
  s.scales = static_cast<const float *>(sc->data);
  s.scale_sh = (int32_t)sc->stride[0];
  s.ws_ml = reinterpret_cast<float *>(wsb + lay.ml_off);
  s.ws_o = reinterpret_cast<float *>(wsb + lay.o_off);
  s.plan_tab = reinterpret_cast<int2 *>(wsb + lay.tab_off);
  s.status = reinterpret_cast<uint32_t *>(wsb);
  s.B = (int32_t)B;
  s.Qmax = (int32_t)Qmax;
  s.Hq = (int32_t)Hq;
  s.Hkv = (int32_t)Hkv;
  s.G = (int32_t)G;
  s.D = (int32_t)D;
  s.page = (int32_t)page;
  s.rows = (int32_t)rows;
  s.rows_pad = (int32_t)rows_pad;
  s.T = T;
  s.P = P;
  s.capacity = (int32_t)cap;
  s.sm_scale = sm_scale;
  s.kv_e5m2 = (o.flags & VAE4_FLAG_KV_E5M2) ? 1 : 0;
  s.hilo = o.hilo_pv;
  s.dev_plan = dev_plan ? 1 : 0;
  s.t_from_len = t_from_len ? 1 : 0;
  s.plan_G = Gp;
  s.plan_N = n_rows;
  if (dev_plan) {
    const int rg_guess = (int)((Qmax * s.G + n_rows - 1) / n_rows);  // row groups at Qmax
    s.plan_W_guess = plan_width_equal((int)B, (int)Hkv, Gp, (int)cap, rg_guess);
    s.plan_np_guess = (int)((cap + s.plan_W_guess - 1) / s.plan_W_guess);
  }

  CombineParams &c = pr->cp;
  memset(&c, 0, sizeof(c));
  c.ws_ml = s.ws_ml;
  c.ws_o = s.ws_o;
  c.out = out->data;
  c.o_sb = out->stride[0];
  c.o_si = out->stride[1];
  c.o_sh = out->stride[2];
  c.seq = s.seq;
  c.seq_sb = s.seq_sb;
  c.seq_has_qlen = has_qlen;
  c.scales = s.scales;
  c.scale_sh = s.scale_sh;
  c.B = s.B;
  c.Qmax = s.Qmax;
  c.Hq = s.Hq;
  c.Hkv = s.Hkv;
  c.G = s.G;
  c.D = s.D;
  c.rows_pad = s.rows_pad;
  c.T = T;
  c.P = dev_plan ? std::max(P, Gp) : P;  // most partitions one stream can have
  c.capacity = s.capacity;
  c.dev_plan = s.dev_plan;
  c.t_from_len = s.t_from_len;
  c.plan_G = Gp;
  c.plan_N = n_rows;
  c.plan_tab = s.plan_tab;
  c.status = s.status;
  c.num_sms = sms;
  return VAE4_OK;
}

// Validation and parameters of the bridge call (kv, block table, lengths and
// scales follow the verify step's rules; outputs are dense FP16 K and V).
int prepare_bridge(const vae4_tensor *kv, const vae4_tensor *bt, const vae4_tensor *seq,
                   const vae4_tensor *sc, const vae4_tensor *ko, const vae4_tensor *vo,
                   uint32_t *status, int32_t flags, vae4::BridgeParams *bp, bool *empty) {
  if (!kv || !bt || !seq || !sc || !ko || !vo) return VAE4_ERR_NULL;
  if ((flags & ~(VAE4_FLAG_KV_E5M2 | VAE4_FLAG_BRIDGE_RAW)) != 0) return VAE4_ERR_OPTIONS;
  if (kv->dtype != VAE4_U8 || bt->dtype != VAE4_I32 || seq->dtype != VAE4_I32 ||
      sc->dtype != VAE4_F32 || ko->dtype != VAE4_F16 || vo->dtype != VAE4_F16)
    return VAE4_ERR_DTYPE;
  if (kv->ndim != 5 || kv->shape[1] != 2 || kv->shape[0] < 1 || kv->shape[2] < 1)
    return VAE4_ERR_SHAPE;
  const int64_t n_pages = kv->shape[0], Hkv = kv->shape[2], page = kv->shape[3], D = kv->shape[4];
  if (D != 64 && D != 128 && D != 256) return VAE4_ERR_UNSUPPORTED;
  if (page < 16 || page % 16 != 0 || page > 65536) return VAE4_ERR_UNSUPPORTED;
  if (kv->stride[4] != 1 || kv->stride[3] != D || kv->stride[2] != page * D ||
      kv->stride[1] != Hkv * page * D || kv->stride[0] != 2 * Hkv * page * D)
    return VAE4_ERR_STRIDE;
  if (!al16(kv->data)) return VAE4_ERR_MISALIGNED;
  // outputs: F16 [B][Hkv][cap][D], d contiguous, rows on 16-byte boundaries
  for (const vae4_tensor *o : {ko, vo}) {
    if (o->ndim != 4 || o->shape[1] != Hkv || o->shape[3] != D || o->shape[2] < 1)
      return VAE4_ERR_SHAPE;
    if (o->shape[0] != ko->shape[0] || o->shape[2] != ko->shape[2]) return VAE4_ERR_SHAPE;
    if (o->stride[3] != 1) return VAE4_ERR_STRIDE;
    for (int k = 0; k < 3; ++k)
      if (o->stride[k] < 0 || o->stride[k] % 8 != 0) return VAE4_ERR_STRIDE;
    if (o->stride[0] != ko->stride[0] || o->stride[1] != ko->stride[1] ||
        o->stride[2] != ko->stride[2])
      return VAE4_ERR_STRIDE;
    if (!al16(o->data)) return VAE4_ERR_MISALIGNED;
  }
  const int64_t B = ko->shape[0], cap = ko->shape[2];
  if (B > 65535 || cap > INT32_MAX / 2) return VAE4_ERR_SHAPE;
  if (bt->ndim != 2 || bt->shape[0] != B || bt->shape[1] < 1) return VAE4_ERR_SHAPE;
  if (bt->stride[1] != 1 || bt->stride[0] < 0) return VAE4_ERR_STRIDE;
  if (bt->shape[1] * page < cap) return VAE4_ERR_SHAPE;  // the table must address cap tokens
  if (seq->ndim == 1) {
    if (seq->shape[0] != B) return VAE4_ERR_SHAPE;
  } else if (seq->ndim == 2) {
    if (seq->shape[0] != B || seq->shape[1] != 2) return VAE4_ERR_SHAPE;
    if (seq->stride[1] != 1) return VAE4_ERR_STRIDE;
  } else {
    return VAE4_ERR_SHAPE;
  }
  if (seq->stride[0] < 0 || seq->stride[0] > INT32_MAX) return VAE4_ERR_STRIDE;
  if (sc->ndim != 2 || sc->shape[0] != Hkv || sc->shape[1] != 2) return VAE4_ERR_SHAPE;
  if (sc->stride[1] != 1 || sc->stride[0] < 0 || sc->stride[0] > INT32_MAX) return VAE4_ERR_STRIDE;
  *empty = B == 0;
  if (B > 0 && (!kv->data || !bt->data || !seq->data || !sc->data || !ko->data || !vo->data))
    return VAE4_ERR_NULL;
  vae4::BridgeParams &p = *bp;
  memset(&p, 0, sizeof(p));
  p.kv = static_cast<const uint8_t *>(kv->data);
  p.n_pages = n_pages;
  p.bt = static_cast<const int32_t *>(bt->data);
  p.bt_sb = bt->stride[0];
  p.seq = static_cast<const int32_t *>(seq->data);
  p.seq_sb = (int32_t)seq->stride[0];
  p.scales = static_cast<const float *>(sc->data);
  p.scale_sh = (int32_t)sc->stride[0];
  p.k_out = static_cast<uint16_t *>(ko->data);
  p.v_out = static_cast<uint16_t *>(vo->data);
  p.o_sb = ko->stride[0];
  p.o_sh = ko->stride[1];
  p.o_st = ko->stride[2];
  p.status = status;
  p.B = (int32_t)B;
  p.Hkv = (int32_t)Hkv;
  p.D = (int32_t)D;
  p.page = (int32_t)page;
  p.cap = (int32_t)cap;
  return VAE4_OK;
}

}  // namespace

extern "C" {

int verify_attn_e4m3_bridge_fp16(const vae4_tensor *kv_pages, const vae4_tensor *block_table,
                                 const vae4_tensor *seq_lens, const vae4_tensor *kv_scales,
                                 const vae4_tensor *k_out, const vae4_tensor *v_out,
                                 uint32_t *dev_status, int32_t flags, vae4_stream stream) {
  vae4::BridgeParams bp;
  bool empty = false;
  int rc = prepare_bridge(kv_pages, block_table, seq_lens, kv_scales, k_out, v_out, dev_status,
                          flags, &bp, &empty);
  if (rc) return rc;
  if (empty) return VAE4_OK;
  int sms = 0;
  rc = device_sms(&sms);
  if (rc) return rc;
  if (vae4::launch_bridge(bp, sms, (flags & VAE4_FLAG_KV_E5M2) != 0,
                          (flags & VAE4_FLAG_BRIDGE_RAW) != 0,
                          reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return VAE4_ERR_CUDA;
  return VAE4_OK;
}

int verify_attn_e4m3_ex(const vae4_tensor *q, const vae4_tensor *kv_pages,
                        const vae4_tensor *block_table, const vae4_tensor *seq_lens,
                        const vae4_tensor *kv_scales, const vae4_tensor *out,
                        const vae4_tensor *workspace, vae4_stream stream,
                        const vae4_options *opt) {
  Prepared pr;
  int rc = prepare(q, kv_pages, nullptr, nullptr, block_table, seq_lens, kv_scales, out,
                   workspace, opt, &pr);
  if (rc) return rc;
  if (pr.empty) return VAE4_OK;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (launch_split(pr, st) != cudaSuccess) return VAE4_ERR_CUDA;
  if (vae4::launch_combine(pr.cp, st) != cudaSuccess) return VAE4_ERR_CUDA;
  return VAE4_OK;
}

int verify_attn_e4m3_kv(const vae4_tensor *q, const vae4_tensor *k_cache,
                        const vae4_tensor *v_cache, const vae4_tensor *block_table,
                        const vae4_tensor *seq_lens, const vae4_tensor *kv_scales,
                        const vae4_tensor *out, const vae4_tensor *workspace,
                        vae4_stream stream, const vae4_options *opt) {
  Prepared pr;
  int rc = prepare(q, nullptr, k_cache, v_cache, block_table, seq_lens, kv_scales, out, workspace,
                   opt, &pr);
  if (rc) return rc;
  if (pr.empty) return VAE4_OK;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (launch_split(pr, st) != cudaSuccess) return VAE4_ERR_CUDA;
  if (vae4::launch_combine(pr.cp, st) != cudaSuccess) return VAE4_ERR_CUDA;
  return VAE4_OK;
}

int verify_attn_e4m3_partials(const vae4_tensor *q, const vae4_tensor *kv_pages,
                              const vae4_tensor *block_table, const vae4_tensor *seq_lens,
                              const vae4_tensor *kv_scales, const vae4_tensor *out,
                              const vae4_tensor *workspace, vae4_stream stream,
                              const vae4_options *opt) {
  Prepared pr;
  int rc = prepare(q, kv_pages, nullptr, nullptr, block_table, seq_lens, kv_scales, out,
                   workspace, opt, &pr);
  if (rc) return rc;
  if (pr.empty) return VAE4_OK;
  if (launch_split(pr, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return VAE4_ERR_CUDA;
  return VAE4_OK;
}

int verify_attn_e4m3_combine(const vae4_tensor *q, const vae4_tensor *kv_pages,
                             const vae4_tensor *block_table, const vae4_tensor *seq_lens,
                             const vae4_tensor *kv_scales, const vae4_tensor *out,
                             const vae4_tensor *workspace, vae4_stream stream,
                             const vae4_options *opt) {
  Prepared pr;
  int rc = prepare(q, kv_pages, nullptr, nullptr, block_table, seq_lens, kv_scales, out,
                   workspace, opt, &pr);
  if (rc) return rc;
  if (pr.empty) return VAE4_OK;
  if (vae4::launch_combine(pr.cp, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return VAE4_ERR_CUDA;
  return VAE4_OK;
}

int verify_attn_e4m3_kv_read(const vae4_tensor *q, const vae4_tensor *kv_pages,
                             const vae4_tensor *block_table, const vae4_tensor *seq_lens,
                             const vae4_tensor *kv_scales, const vae4_tensor *out,
                             const vae4_tensor *workspace, vae4_stream stream,
                             const vae4_options *opt) {
  Prepared pr;
  int rc = prepare(q, kv_pages, nullptr, nullptr, block_table, seq_lens, kv_scales, out,
                   workspace, opt, &pr);
  if (rc) return rc;
  if (pr.empty) return VAE4_OK;
  if (vae4::launch_kv_read(pr.sp, pr.num_sms, reinterpret_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return VAE4_ERR_CUDA;
  return VAE4_OK;
}

int verify_attn_e4m3(const vae4_tensor *q, const vae4_tensor *kv_pages,
                     const vae4_tensor *block_table, const vae4_tensor *seq_lens,
                     const vae4_tensor *kv_scales, const vae4_tensor *out,
                     const vae4_tensor *workspace, vae4_stream stream) {
  return verify_attn_e4m3_ex(q, kv_pages, block_table, seq_lens, kv_scales, out, workspace,
                             stream, nullptr);
}

int verify_attn_e4m3_plan(int B, int Hkv, int max_seq_len, int partition_tokens, int num_sms,
                          int32_t *partition_tokens_out, int32_t *partitions_out) {
  if (!partition_tokens_out || !partitions_out) return VAE4_ERR_NULL;
  int T = 0, P = 0;
  const int rc = do_plan(B, Hkv, max_seq_len, partition_tokens, num_sms, &T, &P);
  if (rc) return rc;
  *partition_tokens_out = T;
  *partitions_out = P;
  return VAE4_OK;
}

int64_t verify_attn_e4m3_workspace_bytes(int B, int Hq, int Hkv, int Qmax, int D,
                                         int max_seq_len, int partition_tokens, int num_sms) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Qmax < 1 || Qmax > kMaxQmax || max_seq_len < 1)
    return VAE4_ERR_SHAPE;
  if (D != 64 && D != 128 && D != 256) return VAE4_ERR_UNSUPPORTED;
  if (Hq % Hkv != 0) return VAE4_ERR_GQA;
  if (align_up((int64_t)Qmax * (Hq / Hkv), 16) > kMaxRowsPad) return VAE4_ERR_UNSUPPORTED;
  const int64_t rows_pad = ws_rows(Qmax * (Hq / Hkv));
  int sms = num_sms;
  if (sms < 0) return VAE4_ERR_SHAPE;
  if (sms == 0) {
    const int rc = device_sms(&sms);
    if (rc) return rc;
  }
  int T = 0, P = 0;
  const int rc = do_plan(B, Hkv, max_seq_len, partition_tokens, sms, &T, &P);
  if (rc) return rc;
  return ws_layout(ws_slots(B, Hkv, P, partition_tokens, sms, vae4_tc_groups(Qmax * (Hq / Hkv))),
                   (int)rows_pad, D, (int64_t)B * Hkv)
      .total;
}

int verify_attn_e4m3_abi_version(void) { return VAE4_ABI_VERSION; }

const char *verify_attn_e4m3_strerror(int code) {
  switch (code) {
    case VAE4_OK: return "ok";
    case VAE4_ERR_NULL: return "a required pointer is NULL";
    case VAE4_ERR_DTYPE: return "wrong dtype";
    case VAE4_ERR_SHAPE: return "inconsistent or out-of-range shape";
    case VAE4_ERR_STRIDE: return "unsupported strides";
    case VAE4_ERR_MISALIGNED: return "base address or row not 16-byte aligned";
    case VAE4_ERR_UNSUPPORTED: return "head dim, page size or row count not supported";
    case VAE4_ERR_GQA: return "q heads not a multiple of KV heads";
    case VAE4_ERR_WORKSPACE: return "workspace too small or not 256-byte aligned";
    case VAE4_ERR_CUDA: return "CUDA runtime error";
    case VAE4_ERR_PARTITION: return "partition_tokens must be a positive multiple of 16 giving at most 8192 partitions";
    case VAE4_ERR_OPTIONS: return "invalid options";
    default: return "unknown error";
  }
}

int verify_attn_e4m3_read_status(const vae4_tensor *workspace, int32_t *host_status,
                                 vae4_stream stream) {
  if (!workspace || !workspace->data || !host_status) return VAE4_ERR_NULL;
  if (workspace->dtype != VAE4_U8) return VAE4_ERR_DTYPE;
  if (workspace->ndim != 1 || workspace->shape[0] < kStatusBytes) return VAE4_ERR_WORKSPACE;
  if (cudaMemcpyAsync(host_status, workspace->data, sizeof(int32_t), cudaMemcpyDeviceToHost,
                      reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return VAE4_ERR_CUDA;
  return VAE4_OK;
}

int verify_attn_e4m3_clear_status(const vae4_tensor *workspace, vae4_stream stream) {
  if (!workspace || !workspace->data) return VAE4_ERR_NULL;
  if (workspace->dtype != VAE4_U8) return VAE4_ERR_DTYPE;
  if (workspace->ndim != 1 || workspace->shape[0] < kStatusBytes) return VAE4_ERR_WORKSPACE;
  if (cudaMemsetAsync(workspace->data, 0, sizeof(int32_t),
                      reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return VAE4_ERR_CUDA;
  return VAE4_OK;
}

int verify_attn_e4m3_decode_table(void *dev_out, int32_t *scale_log2, int32_t flags,
                                  vae4_stream stream) {
  if (!dev_out || !scale_log2) return VAE4_ERR_NULL;
  if (!al16(dev_out)) return VAE4_ERR_MISALIGNED;
  if ((flags & ~(VAE4_FLAG_WARP_MMA | VAE4_FLAG_KV_E5M2)) != 0) return VAE4_ERR_OPTIONS;
  if ((flags & VAE4_FLAG_WARP_MMA) && (flags & VAE4_FLAG_KV_E5M2)) return VAE4_ERR_UNSUPPORTED;
  const bool integer_path = (flags & VAE4_FLAG_WARP_MMA) != 0;
  const bool e5m2 = (flags & VAE4_FLAG_KV_E5M2) != 0;
  *scale_log2 = integer_path ? -8 : 0;
  if (vae4::launch_decode_table(static_cast<uint16_t *>(dev_out), integer_path, e5m2,
                                reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return VAE4_ERR_CUDA;
  return VAE4_OK;
}

}  // extern "C"
