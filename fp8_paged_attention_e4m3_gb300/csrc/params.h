// Launch parameters shared by the host entry points and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace vae4 {

// The device-side balanced plan serves automatic plans of up to this many
// sequences (every CTA scans the batch's lengths).
constexpr int kDevPlanMaxB = 1024;

// Everything a split (partition) kernel needs.  Strides are in elements.
struct SplitParams {
  const void *q;        // fp16 [B][Qmax][Hq][D]
  int64_t q_sb, q_si, q_sh;
  const uint8_t *kv;    // u8 [n_pages][2][Hkv][page][D] (the pool form; null for separate K/V)
  int64_t n_pages;
  // Where token t of KV head h in physical page ph lives, for K and for V:
  // base + ph * ps + (t % page) * ts + h * hs (bytes; d contiguous).  The
  // pool form is one choice of these; the token-major cache another.
  const uint8_t *k_base, *v_base;
  int64_t k_ps, k_ts, k_hs, v_ps, v_ts, v_hs;
  int32_t kv_cpasync;   // 1: strides are multiples of 8 but not all of 16 (8-byte copies)
  const int32_t *bt;    // i32 [B][max_pages]
  int64_t bt_sb;
  int32_t max_pages;
  const int32_t *seq;   // i32 [B] or [B][2]
  int32_t seq_sb;       // stride of dim 0
  int32_t seq_has_qlen; // 1 if [B][2]
  const float *scales;  // f32 [Hkv][2], row stride scale_sh
  int32_t scale_sh;
  float *ws_ml;         // f32 [B][Hkv][P][rows_pad][2]
  float *ws_o;          // f32 [B][Hkv][P][rows_pad][D]
  uint32_t *status;     // sticky status word
  int32_t B, Qmax, Hq, Hkv, G, D, page;
  int32_t rows;         // Qmax * G
  int32_t rows_pad;     // rows rounded up to 16
  int32_t T;            // partition tokens
  int32_t P;            // partitions per (b, h)
  int32_t capacity;     // launch capacity (tokens)
  float sm_scale;       // softmax scale
  int32_t kv_e5m2;      // 1: the KV bytes are E5M2, 0: E4M3
  int32_t dev_plan;     // 1: partitions from the device-side balanced plan (grid.x = G)
  int32_t plan_G;       // device plan: CTAs along x = workspace slots
  int32_t plan_N;       // device plan: rows per CTA (a row group)
  int2 *plan_tab;       // device plan: (first slot, partitions) [B][Hkv], for the combine
  int32_t plan_W_guess, plan_np_guess;  // device plan when every L is the capacity
  int32_t t_from_len;   // static grid: T = max(64, ceil16(L / P)) per sequence
  int32_t hilo;         // 1: P enters the value product as FP16 high + residual
};

// The combine kernel's parameters.
struct CombineParams {
  const float *ws_ml;
  const float *ws_o;
  void *out;            // fp16 [B][Qmax][Hq][D]
  int64_t o_sb, o_si, o_sh;
  const int32_t *seq;
  int32_t seq_sb, seq_has_qlen;
  const float *scales;
  int32_t scale_sh;
  int32_t B, Qmax, Hq, Hkv, G, D;
  int32_t rows_pad, T, P, capacity;
  int32_t dev_plan, plan_G;  // device-side balanced plan and its CTA count
  int32_t plan_N;            // device plan: rows per split CTA
  const int2 *plan_tab;      // device plan: (first slot, partitions) [B][Hkv]
  int32_t t_from_len;        // static grid, T from each sequence's length
  uint32_t *status;
  int32_t num_sms;           // SMs the grid is sized for
};

// The bridge kernel's parameters (paged FP8 -> dense FP16 K and V).
struct BridgeParams {
  const uint8_t *kv;    // u8 [n_pages][2][Hkv][page][D] (the pool form; null for separate K/V)
  int64_t n_pages;
  // Where token t of KV head h in physical page ph lives, for K and for V:
  // base + ph * ps + (t % page) * ts + h * hs (bytes; d contiguous).  The
  // pool form is one choice of these; the token-major cache another.
  const uint8_t *k_base, *v_base;
  int64_t k_ps, k_ts, k_hs, v_ps, v_ts, v_hs;
  int32_t kv_cpasync;   // 1: strides are multiples of 8 but not all of 16 (8-byte copies)
  const int32_t *bt;    // i32 [B][max_pages]
  int64_t bt_sb;
  const int32_t *seq;   // i32 [B] or [B][2] (L first)
  int32_t seq_sb;
  const float *scales;  // f32 [Hkv][2]
  int32_t scale_sh;
  uint16_t *k_out, *v_out;       // fp16 bits [B][Hkv][cap][D]
  int64_t o_sb, o_sh, o_st;      // strides in elements (d stride 1)
  uint32_t *status;     // optional sticky status word (device), may be null
  int32_t B, Hkv, D, page, cap;
};

}  // namespace vae4
