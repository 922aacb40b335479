/*
 * verify_attn_e4m3.h -- C ABI of the GB300 (sm_103a) paged grouped-query
 * verify attention over an FP8 E4M3 KV cache with FP32 split-K state.
 *
 * The operation (sources: the 1Cat-vLLM pull-request pages
 *   PR #560 "[Bugfix] Use FP32 state and E4M3 defaults for DFlash2",
 *   PR #566 "[Kernel] Finalize the audited TP2 DFlash2 31/29 ms endpoint",
 *   PR #524 "[Kernel][SM70] Add opt-in E4M3 grouped attention with FP32
 *            partials"):
 *
 *   For sequence b with L = seq_len[b] cached tokens whose last q = q_len[b]
 *   positions are the draft tokens being verified, query i (0 <= i < q) of q
 *   head hq attends causally to keys 0 .. L-q+i of KV head h = hq / (Hq/Hkv)
 *   (dense q2-8 with 6 q heads per KV head and D = 256, lengths held per
 *   query on the device: PR #524, Scope and non-duplication; q1 and q16 per
 *   PR #560, Purpose and Test Plan):
 *
 *     z_j  = softmax_scale * sum_d Q[b,i,hq,d] * dec(K_j[d]) * s_K[h]
 *     out  = sum_j exp(z_j - max z) * dec(V_j[d]) * s_V[h] / sum_j exp(z_j - max z)
 *
 *   dec() is the exact E4M3 (OCP E4M3FN) decode (PR #566, Final audit);
 *   s_K, s_V are per-KV-head FP32 scales (PR #560, Test Plan and Results).  The KV storage stays FP8 and the tensor
 *   core operands FP16 (PR #560, Purpose).  The context is split into
 *   partitions whose state -- running max, running sum and unnormalised P.V
 *   -- stays FP32 until one final FP32 combine in ascending partition order
 *   (PR #524, final status; PR #560, Purpose).
 *
 * Conventions of every entry point:
 *   - All tensor data pointers are DEVICE pointers unless stated otherwise.
 *     Strides are in elements.  The library never allocates or frees device
 *     memory: the caller owns every buffer, including the workspace.
 *   - Calls are asynchronous on `stream` and never synchronise the host, so
 *     they can be captured in a CUDA graph.  Lengths, block table and scales
 *     are read on the device, so they may change between graph replays.
 *   - A workspace serves one call in flight at a time: use one workspace per
 *     concurrently executing stream (the pages keep separate workspaces per
 *     data type: PR #560, Test Plan and Results).
 *   - Argument errors are returned as negative codes before anything is
 *     launched.  Data errors only visible on the device (block id out of
 *     range, a length beyond capacity, q_len > L, a bounded wait that ran
 *     out) set bits in a sticky status word inside the workspace and zero
 *     the affected sequence's output; nothing traps or aborts.
 */
#ifndef VERIFY_ATTN_E4M3_H_
#define VERIFY_ATTN_E4M3_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ABI revision.  A wrapper refuses a library whose revision differs from the
 * one it was written for, so an out-of-date library is refused rather than
 * used (PR #524, Scope and non-duplication; PR #560, Purpose). */
#define VAE4_ABI_VERSION 2

/* Same object as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *vae4_stream;

enum vae4_dtype {
  VAE4_U8 = 1,  /* E4M3 bytes */
  VAE4_I32 = 2,
  VAE4_F16 = 3,
  VAE4_F32 = 4
};

/* A strided view.  `data` is a device pointer unless an entry point says
 * otherwise; shape/stride entries beyond ndim are ignored. */
typedef struct {
  void *data;
  int32_t dtype; /* enum vae4_dtype */
  int32_t ndim;
  int64_t shape[5];
  int64_t stride[5]; /* elements */
} vae4_tensor;

/* Optional parameters of verify_attn_e4m3_ex (zero-initialise for defaults). */
typedef struct {
  float softmax_scale;      /* 0 -> 1/sqrt(D) */
  int32_t partition_tokens; /* split-K partition length T (multiple of 16);
                               0 -> automatic plan, made on the device from
                               the lengths of the call (see
                               verify_attn_e4m3_plan) */
  int32_t max_seq_len;      /* launch capacity in tokens; 0 ->
                               block_table columns * page size */
  int32_t num_sms;          /* SMs the plan targets; 0 -> current device */
  int32_t flags;            /* 0, or VAE4_FLAG_WARP_MMA / VAE4_FLAG_KV_E5M2 */
  int32_t hilo_pv;          /* 1 -> P enters the value product as an FP16
                               high part and an FP16 residual scaled by 2^11
                               (see below); 0 -> one FP16 P */
} vae4_options;

/* hilo_pv: the high/residual representation of the softmax probabilities
 * in the value product (PR #524 "[Kernel][SM70] Add opt-in E4M3 grouped
 * attention with FP32 partials", Historical R6 purpose and evidence, Scope
 * and non-duplication: the residual is multiplied by 2048 and its product
 * scaled back by the exactly representable 1/2048).  With p the FP32
 * probability, P_hi = fp16(p) and P_lo = fp16((p - P_hi) * 2^11); the
 * partition accumulates P_hi.V + 2^-11 P_lo.V in FP32 and its running sum
 * adds the same P_hi + 2^-11 P_lo, so P carries ~22 significant bits into
 * the FP32 state instead of 11.  The kernel forms both parts from 2^11 p
 * (so both products share one accumulator) and therefore raises its lazy
 * running maximum at 2^4 instead of 2^12, which keeps 2^11 p inside FP16.
 * It costs a second value MMA per key step and more running-maximum
 * updates.  Only the default tcgen05 path implements it: with
 * VAE4_FLAG_WARP_MMA the call returns VAE4_ERR_UNSUPPORTED. */

/* Option flag: run the split stage on the warp-level tensor-core path
 * (mma.sync m16n8k16 with ldmatrix operands) instead of the default
 * tcgen05 / TMEM / TMA kernel.  Same contract and precision; kept as the
 * measured legacy baseline. */
#define VAE4_FLAG_WARP_MMA 0x1

/* Option flag: the KV bytes are OCP FP8 E5M2 (sign, 5-bit exponent with
 * bias 15, 2-bit mantissa; largest finite value 57344) instead of E4M3.
 * The pages keep the E5M2 cache format available beside E4M3 (PR #560,
 * Purpose; PR #524, Scope and non-duplication).  Every finite E5M2 value is
 * an FP16 value, so the decode stays exact; scales, state and combine are
 * unchanged.  The infinity and NaN codes are outside the contract.  Only the
 * default tcgen05 path implements it: with VAE4_FLAG_WARP_MMA the call
 * returns VAE4_ERR_UNSUPPORTED. */
#define VAE4_FLAG_KV_E5M2 0x2

/* Test hook for the failure path: every pipeline wait of the tcgen05 split
 * kernel gives up after ~256 SM cycles instead of ~1 s, so the call aborts
 * the way a stalled pipeline would (no fault: copies and MMAs in flight are
 * still drained before the CTA exits), reports VAE4_STATUS_TIMEOUT and
 * writes zero rows.  Not for production use; VAE4_ERR_UNSUPPORTED together
 * with VAE4_FLAG_WARP_MMA. */
#define VAE4_FLAG_TEST_SHORT_WAITS 0x8

/* Bridge flag: write dec(byte) without the per-head scale (exact). */
#define VAE4_FLAG_BRIDGE_RAW 0x4

/* Return codes. */
enum vae4_error {
  VAE4_OK = 0,
  VAE4_ERR_NULL = -1,        /* a required pointer is NULL */
  VAE4_ERR_DTYPE = -2,       /* a tensor has the wrong dtype */
  VAE4_ERR_SHAPE = -3,       /* inconsistent or out-of-range shapes */
  VAE4_ERR_STRIDE = -4,      /* unsupported strides (see each argument) */
  VAE4_ERR_MISALIGNED = -5,  /* a base address or row is not 16-byte aligned */
  VAE4_ERR_UNSUPPORTED = -6, /* D, page size or rows outside the kernels' set */
  VAE4_ERR_GQA = -7,         /* Hq is not a multiple of Hkv */
  VAE4_ERR_WORKSPACE = -8,   /* workspace too small or misaligned */
  VAE4_ERR_CUDA = -9,        /* a CUDA runtime call failed */
  VAE4_ERR_PARTITION = -10,  /* partition_tokens not a positive multiple of 16,
                                or more than 8192 partitions per sequence */
  VAE4_ERR_OPTIONS = -11     /* unknown option flags or a negative scale */
};

/* Bits of the device status word (sticky until verify_attn_e4m3_clear_status). */
#define VAE4_STATUS_BAD_BLOCK 0x1u  /* block id < 0 or >= number of pages */
#define VAE4_STATUS_BAD_LENGTH 0x2u /* L < 0 or L > launch capacity */
#define VAE4_STATUS_BAD_QLEN 0x4u   /* q_len < 0, q_len > Qmax, or q_len > L > 0 */
#define VAE4_STATUS_TIMEOUT 0x8u    /* a bounded pipeline wait ran out */
#define VAE4_STATUS_PLAN 0x10u      /* a stream's record of the device-side plan is out of
                                       range (an internal invariant; the rows are zeroed) */

/*
 * verify_attn_e4m3 -- the verify step (split kernel + combine kernel).
 *
 *  q           F16 [B][Qmax][Hq][D]; D in {64, 128, 256}; Qmax <= 16;
 *              stride[3] == 1, other strides multiples of 8 elements, base
 *              16-byte aligned (a misaligned view is rejected, never copied;
 *              cf. the Q-base safety repair of PR #524, final status).  Slot
 *              i of sequence b is a query only if i < q_len[b]; the other
 *              slots are padding and are never read.
 *  kv_pages    U8 [n_pages][2][Hkv][page][D], contiguous; index 0 of dim 1
 *              is K, 1 is V; page = any multiple of 16 tokens up to 65536
 *              (the pages run 16-token pages and 848- to 3456-token blocks:
 *              PR #560, Purpose and Test Plan and Results; PR #524, AI
 *              review); base 16-byte aligned.  Each (page, K|V, head) slice
 *              of page*D bytes is one contiguous 16-byte-aligned block.
 *              Slots past L in a sequence's last page may hold anything
 *              (e.g. never written, NaN codes): they do not reach the
 *              output.
 *  block_table I32 [B][max_pages], stride[1] == 1: logical page j of
 *              sequence b lives in physical page block_table[b][j].  The ids
 *              of the first ceil(L/page) entries of a row are used; up to 64
 *              entries beyond them (within the row) may be read and ignored.
 *  seq_lens    I32 [B] (L; q_len = Qmax for every sequence) or I32 [B][2]
 *              with stride[1] == 1 holding (L, q_len).  L counts the q tail.
 *              L == 0 marks a dead sequence (all-zero output, no status bit).
 *  kv_scales   F32 [Hkv][2] = (s_K, s_V), stride[1] == 1.
 *  out         F16, same shape as q, same stride rules; written in full
 *              (padding slots and dead sequences get zeros).  Must not
 *              overlap any input.
 *  workspace   U8 [bytes], bytes >= verify_attn_e4m3_workspace_bytes(...),
 *              base 256-byte aligned.  Holds the FP32 partials and the
 *              status word.  Zero-fill it (or call
 *              verify_attn_e4m3_clear_status) once before first use.
 *  stream      CUDA stream of the current device.
 *
 * Returns VAE4_OK or a negative vae4_error; on error nothing is launched.
 */
int verify_attn_e4m3(const vae4_tensor *q, const vae4_tensor *kv_pages,
                     const vae4_tensor *block_table, const vae4_tensor *seq_lens,
                     const vae4_tensor *kv_scales, const vae4_tensor *out,
                     const vae4_tensor *workspace, vae4_stream stream);

/* As verify_attn_e4m3, with options (NULL = defaults). */
int verify_attn_e4m3_ex(const vae4_tensor *q, const vae4_tensor *kv_pages,
                        const vae4_tensor *block_table, const vae4_tensor *seq_lens,
                        const vae4_tensor *kv_scales, const vae4_tensor *out,
                        const vae4_tensor *workspace, vae4_stream stream,
                        const vae4_options *opt);

/*
 * verify_attn_e4m3_kv -- the verify step over separate K and V caches in
 * any strided layout, e.g. the token-major [blocks][block_size][kv_heads]
 * [head_dim] caches of the pages, including padded token strides that are
 * multiples of 8 but not of 16 bytes (the [1,848,1,256] view with strides
 * [223872,264,256,1] of PR #524 "[Kernel][SM70] Add opt-in E4M3 grouped
 * attention with FP32 partials", AI integration review and revision-2
 * update).
 *
 *  k_cache, v_cache  U8 [n_pages][page][Hkv][D], the same shape; stride[3]
 *              == 1; the other strides (in bytes, any order, K and V may
 *              differ) non-negative multiples of 8; bases 8-byte aligned;
 *              page = any multiple of 16 tokens up to 65536.  Token t of
 *              sequence b, KV head h is k_cache[block_table[b][t / page]]
 *              [t % page][h][:], and likewise in v_cache.
 *  Other arguments, options, results and errors as verify_attn_e4m3_ex.
 *
 * When both caches have 16-byte aligned bases and strides that are
 * multiples of 16 bytes (e.g. a contiguous token-major cache), their page
 * slices are moved by tensor copies as for the pool; otherwise by 8-byte
 * asynchronous copies (slower, same results).  The legacy mma.sync path
 * (VAE4_FLAG_WARP_MMA) reads only the pool form: VAE4_ERR_UNSUPPORTED.
 */
int verify_attn_e4m3_kv(const vae4_tensor *q, const vae4_tensor *k_cache,
                        const vae4_tensor *v_cache, const vae4_tensor *block_table,
                        const vae4_tensor *seq_lens, const vae4_tensor *kv_scales,
                        const vae4_tensor *out, const vae4_tensor *workspace,
                        vae4_stream stream, const vae4_options *opt);

/*
 * The two stages of verify_attn_e4m3, for callers that schedule them apart
 * (e.g. to time or overlap them).  Same arguments and contract.
 *   verify_attn_e4m3_partials: the split kernel only -- writes each live
 *     partition's FP32 (max, sum, unnormalised P.V) into the workspace.
 *   verify_attn_e4m3_combine: the combine kernel only -- reads the partials
 *     of the same arguments from the workspace and writes `out`.  It must
 *     follow a verify_attn_e4m3_partials call with identical arguments on
 *     the same stream; q and kv_pages are not read.
 */
int verify_attn_e4m3_partials(const vae4_tensor *q, const vae4_tensor *kv_pages,
                              const vae4_tensor *block_table,
                              const vae4_tensor *seq_lens,
                              const vae4_tensor *kv_scales, const vae4_tensor *out,
                              const vae4_tensor *workspace, vae4_stream stream,
                              const vae4_options *opt);
int verify_attn_e4m3_combine(const vae4_tensor *q, const vae4_tensor *kv_pages,
                             const vae4_tensor *block_table,
                             const vae4_tensor *seq_lens,
                             const vae4_tensor *kv_scales, const vae4_tensor *out,
                             const vae4_tensor *workspace, vae4_stream stream,
                             const vae4_options *opt);

/*
 * verify_attn_e4m3_bridge_fp16 -- the explicit paged-FP8 -> FP16 bridge the
 * pages describe next to the grouped attention (PR #524 "[Kernel][SM70] Add
 * opt-in E4M3 grouped attention with FP32 partials", historical R6 purpose
 * and scope): the cache's decode and page gather as a call of its own.
 *
 *  kv_pages, block_table, seq_lens, kv_scales: as for verify_attn_e4m3
 *              (seq_lens I32 [B] or [B][2]; only L is used).
 *  k_out, v_out F16 [B][Hkv][cap][D], stride[3] == 1, other strides
 *              multiples of 8 elements (equal for both), 16-byte aligned;
 *              block_table must address cap tokens (columns * page >= cap).
 *  dev_status  optional device pointer to a status word (NULL = none):
 *              VAE4_STATUS_BAD_BLOCK / BAD_LENGTH bits are OR-ed in.
 *  flags       VAE4_FLAG_KV_E5M2 (bytes are E5M2), VAE4_FLAG_BRIDGE_RAW.
 *
 * For every sequence b with 0 <= L <= cap and KV head h, token t < L:
 *   k_out[b][h][t][:] = fp16(dec(K byte) * s_K[h]), v_out likewise with s_V,
 * each rounded once (to nearest even) from the exact product; with
 * VAE4_FLAG_BRIDGE_RAW, fp16(dec(byte)) (exact, no scale).  Tokens t >= L
 * are not written.  A page with an invalid id writes zeros for its tokens
 * and sets BAD_BLOCK; L > cap skips the sequence and sets BAD_LENGTH.
 * Asynchronous on `stream`; allocates nothing.
 */
int verify_attn_e4m3_bridge_fp16(const vae4_tensor *kv_pages, const vae4_tensor *block_table,
                                 const vae4_tensor *seq_lens, const vae4_tensor *kv_scales,
                                 const vae4_tensor *k_out, const vae4_tensor *v_out,
                                 uint32_t *dev_status, int32_t flags, vae4_stream stream);

/*
 * Measurement helper (not a step of the method): reads every KV byte that
 * verify_attn_e4m3 with the same arguments reads -- K and V of tokens
 * 0 .. L-1 of every (sequence, KV head), through the block table, in the
 * same page order -- with plain 16-byte loads and no arithmetic.  Its time
 * is the floor of the step's page gather on the running GPU; the pages time
 * their kernels in graph-replayed A/B blocks against a reference in the same
 * way (PR #560 "[Bugfix] Use FP32 state and E4M3 defaults for DFlash2", Test
 * Plan and Results).  Same arguments and validation as verify_attn_e4m3_ex;
 * q and out are validated but not read or written.  XORs every 32-bit word
 * it reads into the word at workspace byte 128 (a checksum: zero that word
 * first to read it; the status word at byte 0 is not touched).  Pages with invalid ids and sequences with invalid lengths are
 * skipped without a status bit.
 */
int verify_attn_e4m3_kv_read(const vae4_tensor *q, const vae4_tensor *kv_pages,
                             const vae4_tensor *block_table,
                             const vae4_tensor *seq_lens,
                             const vae4_tensor *kv_scales, const vae4_tensor *out,
                             const vae4_tensor *workspace, vae4_stream stream,
                             const vae4_options *opt);

/*
 * verify_attn_e4m3_plan -- the split-K partition plan (host only, no CUDA).
 * Partition p of every sequence covers tokens [p*T, min((p+1)*T, L)); the
 * launch has P = ceil(max_seq_len / T) partitions per (sequence, KV head).
 * With partition_tokens == 0, T is the smallest multiple of 16 for which
 * B*Hkv*P does not exceed max(num_sms, B*Hkv) (one wave on the SMs; the
 * pages' split used one partition per V100 SM: the 80 of the [80,8,6,2]
 * workspace, PR #524, final status).  num_sms must be > 0.
 * Returns VAE4_OK, VAE4_ERR_SHAPE or VAE4_ERR_PARTITION.
 *
 * That is the plan for sequences at the capacity.  A call with
 * partition_tokens == 0 refines it on the device from the lengths it reads
 * (so a captured graph stays balanced as the lengths change):
 *  - B == 1 (or B > 1024): each sequence keeps the P partitions above and
 *    takes T = max(64, ceil(L / P) rounded up to 16) from its own L;
 *  - 1 < B <= 1024 (and B*Hkv*row groups <= 65535): the device-side
 *    balanced plan.  One length W, a multiple of 16 and at least 64, for
 *    every (sequence, KV head) stream, P_b = ceil(L_b / W) partitions, each
 *    run by r_b CTAs, one per row group of the split kernel holding a live
 *    query (r_b = ceil(q_len * Hq/Hkv / rows per CTA)), with
 *    sum_b Hkv * r_b * P_b <= G = max(num_sms, B*Hkv*row groups): W from
 *    ceil(sum r L / (G / Hkv)) and at most six bisection steps.  All live
 *    CTAs run in one wave; partitions are numbered by r_b (largest first),
 *    then sequence, KV head and partition.
 * Both give the same results as any fixed T up to FP32 rounding order.
 */
int verify_attn_e4m3_plan(int B, int Hkv, int max_seq_len, int partition_tokens,
                          int num_sms, int32_t *partition_tokens_out,
                          int32_t *partitions_out);

/*
 * verify_attn_e4m3_workspace_bytes -- bytes of workspace a call with these
 * sizes needs: the status word, FP32 (max, sum) per partition and row
 * ([B][Hkv][P][rows][2], the pages' [80,8,6,2] "max/sum" layout, PR #524,
 * final status) and the FP32 unnormalised P.V per partition and row
 * ([B][Hkv][P][rows][D]); rows = Qmax * Hq/Hkv rounded up to 16.  With
 * partition_tokens == 0 and 1 < B <= 1024 the partials take
 * max(B*Hkv*P, num_sms, B*Hkv*row groups) slots of [rows] (the device
 * plan's grid); a final B*Hkv*8 bytes hold each stream's (first slot,
 * partitions) under that plan.
 * num_sms == 0 queries the current device (a CUDA call); any other value
 * makes this a pure host computation.  Returns the size, or a negative
 * vae4_error.
 */
int64_t verify_attn_e4m3_workspace_bytes(int B, int Hq, int Hkv, int Qmax, int D,
                                         int max_seq_len, int partition_tokens,
                                         int num_sms);

/* VAE4_ABI_VERSION of the built library. */
int verify_attn_e4m3_abi_version(void);

/* Static string for a vae4_error code. */
const char *verify_attn_e4m3_strerror(int code);

/* Copy the status word of `workspace` into *host_status (host pointer) with
 * an asynchronous copy on `stream`; read it after synchronising the stream. */
int verify_attn_e4m3_read_status(const vae4_tensor *workspace,
                                 int32_t *host_status, vae4_stream stream);

/* Zero the status word of `workspace` on `stream`. */
int verify_attn_e4m3_clear_status(const vae4_tensor *workspace, vae4_stream stream);

/*
 * verify_attn_e4m3_decode_table -- test hook for the exact decoders: runs a
 * split kernel's E4M3 -> FP16 decode routine on all 256 byte codes and
 * writes the raw FP16 bit patterns to dev_out (device, 256 x uint16).
 * flags selects the kernel as in vae4_options.flags: 0 = the tcgen05 path
 * (hardware converter, dec(b) exactly), VAE4_FLAG_WARP_MMA = the mma.sync
 * path (integer bit move, dec(b) * 2^-8 exactly), VAE4_FLAG_KV_E5M2 = the
 * tcgen05 path's E5M2 decode (byte move, dec(b) exactly, infinities and
 * NaNs as in FP16).  *scale_log2 (host
 * pointer) receives the exponent e with FP16 = dec(b) * 2^e; the kernels
 * fold 2^-e into their FP32 scales.  The NaN codes 0x7F / 0xFF are outside
 * the contract (NaN on the first decoder, a finite pattern on the second).
 * (The pages test the decoder on every E4M3 byte: PR #566, Test Result.)
 */
int verify_attn_e4m3_decode_table(void *dev_out, int32_t *scale_log2, int32_t flags,
                                  vae4_stream stream);

/* Bytes of the library-owned scratch that verify_attn_e4m3_noalloc uses. */
#define VAE4_NOALLOC_SCRATCH_BYTES (8u << 20)

/*
 * verify_attn_e4m3_noalloc -- the verify step for callers that cannot
 * allocate device memory.  (No counterpart on the pages: this is an
 * addition of this library.)
 *
 * Some callers have no way to hand over a workspace: code that runs where a
 * device allocation is forbidden or unsafe -- inside a region being
 * captured into a CUDA graph, inside a plugin or custom-op callback whose
 * host framework owns all device memory and gives none out at execution
 * time, or in a serving loop with a fixed memory budget where cudaMalloc
 * could block on the device or fail under fragmentation.  This entry point
 * takes the same arguments as verify_attn_e4m3_ex without the workspace:
 * the FP32 partials and the status word live in a fixed scratch array of
 * VAE4_NOALLOC_SCRATCH_BYTES (8 MiB) that the library declares statically,
 * so every GPU that loads the library keeps those 8 MiB reserved until the
 * process exits.  Nothing is allocated or freed: no cudaMalloc, no
 * cudaFree, no allocating library routine.
 *
 *  - The first call on a device looks up the scratch array's device
 *    address (once per device, with that device current; again after
 *    cudaDeviceReset, which makes a new context).  Make that first call
 *    before any stream capture on the device.
 *  - A call whose partition plan needs more than VAE4_NOALLOC_SCRATCH_BYTES
 *    (see verify_attn_e4m3_workspace_bytes) returns VAE4_ERR_WORKSPACE and
 *    launches nothing.  Example sizes: the 262144-token q8 GQA6 D256 step
 *    on 152 SMs needs about 7.2 MiB.
 *  - Every call on a device shares the one scratch array and leaves its
 *    contents behind.  Nothing in it has to start at zero (each call writes
 *    every partial it reads), so no clearing is done.  Calls whose kernels
 *    overlap on the GPU (different streams without ordering) race on the
 *    scratch and give wrong results: order them.
 *  - Device-side data errors zero the affected sequence's output exactly as
 *    in verify_attn_e4m3_ex; the status word is not readable from here.
 * Returns VAE4_OK or a negative vae4_error.
 */
int verify_attn_e4m3_noalloc(const vae4_tensor *q, const vae4_tensor *kv_pages,
                             const vae4_tensor *block_table,
                             const vae4_tensor *seq_lens,
                             const vae4_tensor *kv_scales, const vae4_tensor *out,
                             vae4_stream stream, const vae4_options *opt);

#ifdef __cplusplus
}
#endif
#endif /* VERIFY_ATTN_E4M3_H_ */
