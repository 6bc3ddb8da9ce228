/*
 * attn.h — C ABI of the GB300 (sm_103a) fused exact-attention forward library
 * (libattn_gb300.so).
 *
 * The operation, from the pages this library follows:
 *   O = softmax(scale * Q K^T [+ causal mask]) V, plus the per-row log-sum-exp (LSE),
 *   computed tile by tile with a running (online) softmax so the N x N score matrix is never
 *   written to memory.
 *   - Formula: "FlashAttention-3 Deep Dive: WGMMA Async Pipelines, FP8 Tensor Cores & GPU Kernel
 *     Optimization in 2026" (mojostudio.in), introduction (softmax(Q K^T / sqrt(d_k)) V) and
 *     section 3 (P_ij = exp(S_ij - m_i)).
 *   - Tiling + running softmax, no N x N in memory: "flash-attention-3" (ai.thesatyajit.com),
 *     opening paragraph.
 *   - Call shape flash_attn_func(q, k, v, causal=True) with q of shape (B, N, H, D):
 *     "Lecture 9 — Hopper / FlashAttention-3 / FlashAttention-4", "Benchmark task".
 *   - GQA and FP8 forward with per-tensor descale factors: "flash-attention-3", "What is
 *     actually in the box" and "FP8 is a different kernel"; "Lecture 9", "FP8".
 *   - LSE: the "Hopper" tag page (l1-ca0.github.io) names it in its section 4.6 title
 *     ("rescaling, correction, and LSE"); read here as the natural-log log-sum-exp of the
 *     scaled, masked scores of the row.
 *
 * All entry points are plain C; pointers are raw device or host addresses as stated per call.
 */
#ifndef GB300_ATTN_H
#define GB300_ATTN_H

#include <stdint.h>
#include <cuda_runtime_api.h> /* cudaStream_t */

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1, /* bad pointer, size, alignment or overlap; nothing was launched   */
  ATTN_ERR_UNSUPPORTED = 2, /* valid request the library does not implement; nothing launched */
  ATTN_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed (launch, copy, sync, no GPU)  */
  ATTN_ERR_TIMEOUT = 4      /* a kernel's bounded wait gave up (reported by attn_get_status)   */
} attn_status_t;

typedef enum {
  ATTN_DTYPE_BF16 = 0,      /* q, k, v are bfloat16                                          */
  ATTN_DTYPE_FP8_E4M3 = 1   /* q, k, v are float8 e4m3 (OCP "fn": max 448) with fp32 descales */
} attn_dtype_t;

/*
 * attn_fwd — fused attention forward on the GPU, asynchronous on `stream`.
 *
 * Arguments (all tensors contiguous, row-major, in DEVICE memory owned by the caller):
 *   q      [B, N, H,   d]  element type `dtype`
 *   k, v   [B, N, Hkv, d]  element type `dtype`; query head h reads kv head h / (H / Hkv)
 *   o      [B, N, H,   d]  bfloat16 output
 *   lse    [B, H, N]       float32 output, LSE_i = ln sum_j exp(scale * q_i . k_j) over the
 *                          keys row i may see (all keys, or j <= i when causal)
 *   B, H, Hkv, N >= 1, H % Hkv == 0; d in {64, 128, 256} for bf16 and for fp8.
 *   scale  finite, nonzero float multiplying the raw dot products (usually 1/sqrt(d)); it does
 *          not include the fp8 descales. A negative scale is allowed (the kernel computes
 *          |scale| * (-Q) K^T, so the softmax's running maximum is taken over the scaled scores
 *          either way). scale == 0 returns ATTN_ERR_UNSUPPORTED: masked scores are -inf before
 *          scaling, and 0 * -inf has no value.
 *   causal nonzero: key j is visible to query i iff j <= i (top-left aligned).
 *   descale_q/k/v  fp8 only: DEVICE pointers to one float each; the value the kernel uses
 *          for an element x8 is x8 * descale. Ignored (may be NULL) for bf16.
 *   stream CUDA stream (0 = legacy default stream).
 *
 * Alignment: q, k, v, o must be 16-byte aligned (tensor-memory-accelerator copies and 16-byte
 * stores); lse 4-byte aligned. o and lse must not overlap q, k, v or each other.
 *
 * Launches: one persistent kernel, one CTA per SM, each CTA walking work tiles of 256 (d <= 128)
 * or 128 (d == 256) query rows of one (batch, head). Non-causal calls whose last wave of work
 * tiles would leave SMs idle cut the key range of some tiles in two (see attn_fwd_tail_units)
 * and make a second launch: the first launch covers each such tile's first keys and writes its
 * O and LSE as usual; the second, a programmatic dependent launch whose CTAs start on the SMs the
 * first one leaves, covers the rest of the keys, waits for the first launch to finish, and merges
 * the two parts into o and lse (LSE = ln(e^LSE_a + e^LSE_b), O = e^(LSE_a - LSE) O_a +
 * e^(LSE_b - LSE) O_b). The first part's O passes through o in bf16, so those rows carry one
 * extra bf16 rounding of that part. Which tiles are cut (T work tiles, G SMs, K = ceil(N / 128)
 * key tiles):
 *   - bf16 at d <= 128, T > G, T not a multiple of G, K >= 8: the tiles after the first
 *     M = (floor(T / G) - 1) G go to the CTAs in G equal shares of their W = (T - M) K key
 *     tiles (share c: [floor(c W / G), floor((c + 1) W / G)), counting key tile j of tile M + i
 *     as i K + j), so every CTA processes the same number of key tiles; a tile a share boundary
 *     falls inside is cut there;
 *   - otherwise, when the last wave holds R <= G / 2 tiles and K >= 16: those R tiles, at key
 *     tile floor(K / 2).
 *
 * Errors: argument problems return ATTN_ERR_INVALID_ARG / ATTN_ERR_UNSUPPORTED synchronously
 * and launch nothing. A failed launch returns ATTN_ERR_CUDA. A kernel that gives up a bounded
 * internal wait finishes early and records it in a device status word: read it with
 * attn_get_status. The library allocates no memory in this call and keeps no per-call state.
 */
attn_status_t attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                       int B, int H, int Hkv, int N, int d, float scale, int causal,
                       attn_dtype_t dtype, const float* descale_q, const float* descale_k,
                       const float* descale_v, cudaStream_t stream);

/*
 * attn_fwd_halved_tail_tiles — how many work tiles of a bf16 attn_fwd call have their key range
 * cut in two across two launches, by the rule under attn_fwd's "Launches" (work tiles:
 * B * H * ceil(N / R), R = 256 for d <= 128, 128 for d == 256); attn_fwd_tail_units gives the
 * count for either dtype. 0 means one launch. Host-only; uses 152 SMs when no device can be
 * queried; returns 0 for invalid sizes.
 */
int attn_fwd_halved_tail_tiles(int B, int H, int N, int d, int causal);

/*
 * attn_fwd_tail_units — the cut tiles themselves of an attn_fwd call of this dtype (the e4m3
 * entry points with per-head or block descales follow the e4m3 rule), in the second launch's
 * order: for unit u, tiles[u] is the work tile and kv0[u] the first key tile (of 128 keys) the
 * second launch covers for it. Work tile t of a non-causal call is query block t % n_mb of
 * (batch, head) ((t / n_mb) / H, (t / n_mb) % H), n_mb = ceil(N / R). Writes at most cap units
 * into the HOST arrays tiles and kv0 (either may be NULL when cap is 0) and returns the unit
 * count (0: one launch; also for invalid sizes or dtype). Host-only.
 */
int attn_fwd_tail_units(int B, int H, int N, int d, int causal, attn_dtype_t dtype, int* tiles, int* kv0,
                        int cap);

/*
 * attn_fwd_fp8_scaled — attn_fwd for e4m3 q, k, v with descale factors that vary by batch and
 * head instead of one per tensor. The value used for an element of q in batch b, query head h
 * is x8 * descale_q[b * q_stride_b + h * q_stride_h]; for k and v in batch b, kv head g it is
 * x8 * descale_{k,v}[b * kv_stride_b + g * kv_stride_h]. Strides are in elements (>= 0); all 0
 * reproduces the per-tensor attn_fwd. Per-head scales keep more of e4m3's few mantissa bits when
 * heads differ in magnitude: "flash-attention-3" (ai.thesatyajit.com), "FP8 is a different
 * kernel" (descale pointers with strides).
 *   descale arrays: DEVICE fp32, large enough for every (b, head) the strides address.
 *   Everything else as attn_fwd with dtype ATTN_DTYPE_FP8_E4M3 (d == 64, 128 or 256).
 */
attn_status_t attn_fwd_fp8_scaled(const void* q, const void* k, const void* v, void* o,
                                  float* lse, int B, int H, int Hkv, int N, int d, float scale,
                                  int causal, const float* descale_q, int q_stride_b,
                                  int q_stride_h, const float* descale_k, const float* descale_v,
                                  int kv_stride_b, int kv_stride_h, cudaStream_t stream);

/*
 * Ragged batches ("varlen"): B sequences packed along the row dimension, described by
 * cumulative offsets. Sequence b owns query rows cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 of
 * q [total_q, H, d] and key rows cu_seqlens_k[b] .. cu_seqlens_k[b+1]-1 of k, v [total_k, Hkv, d];
 * query and key lengths may differ and may be 0. "flash-attention-3" (ai.thesatyajit.com),
 * "What is actually in the box" and "Five schedulers"; "FlashAttention-3 Deep Dive"
 * (mojostudio.in), FAQ on variable-length sequences (cu_seqlens, no padding).
 *
 * Causal masking is bottom-right aligned: query i of a sequence with Nq queries and Nk keys sees
 * keys j <= i + (Nk - Nq), so the last query sees every key; with Nq == Nk this is the usual mask.
 * A query row that sees no key (Nk == 0, or i + Nk - Nq < 0) gets O = 0 and LSE = -inf.
 *
 * attn_varlen_plan — builds the work-tile plan of a ragged batch on the GPU (one small kernel on
 * `stream`): every (sequence, query head, block of query rows) tile, longest first. A plan
 * depends on the offsets, B, H, d (through the tile height), causal and the totals, and can be
 * reused by every forward call with the same batch (e.g. all layers of one step).
 *   cu_seqlens_q, cu_seqlens_k: DEVICE int32 [B + 1], starting at 0, non-decreasing, last entry
 *       <= total_q / total_k. Offsets that break this give a plan marked invalid (a forward
 *       handed it writes nothing and attn_get_status reports ATTN_ERR_INVALID_ARG).
 *   plan: DEVICE, 16-byte aligned, plan_bytes >= attn_varlen_plan_bytes(B, H, total_q, d).
 * INVALID_ARG for null or misaligned pointers, negative sizes or a short buffer; UNSUPPORTED for
 * d not in {64, 128, 256}.
 */
size_t attn_varlen_plan_bytes(int B, int H, int total_q, int d);
attn_status_t attn_varlen_plan(const int* cu_seqlens_q, const int* cu_seqlens_k, int B, int H,
                               int total_q, int total_k, int d, int causal, void* plan,
                               size_t plan_bytes, cudaStream_t stream);

/*
 * attn_fwd_varlen — attn_fwd over a ragged batch, asynchronous on `stream`, allocates nothing.
 *   q [total_q, H, d], k, v [total_k, Hkv, d]: DEVICE, element type `dtype`, 16-byte aligned.
 *   o [total_q, H, d] bf16 (DEVICE, 16-byte aligned), lse [H, total_q] fp32 (natural log).
 *   cu_seqlens_q, cu_seqlens_k: DEVICE int32 [B + 1] as for attn_varlen_plan.
 *   plan, plan_bytes: built by attn_varlen_plan from the same offsets, B, H, d, causal, total_q
 *         and total_k, and the size of its buffer. A plan built for other arguments is detected
 *         on the GPU (nothing is written, and attn_get_status reports ATTN_ERR_INVALID_ARG); so
 *         is a tile whose sequence's rows fall outside the packed tensors (that tile is skipped).
 *   descale_q/k/v: e4m3 only, one fp32 each (per tensor), as in attn_fwd.
 * Same argument checks as attn_fwd; total_q == 0 returns ATTN_OK at once.
 */
attn_status_t attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                              const int* cu_seqlens_q, const int* cu_seqlens_k, const void* plan,
                              size_t plan_bytes, int B, int H, int Hkv, int total_q, int total_k,
                              int d, float scale, int causal, attn_dtype_t dtype,
                              const float* descale_q, const float* descale_k,
                              const float* descale_v, cudaStream_t stream);

/*
 * attn_bwd — gradients of attn_fwd (bf16, d in {64, 128}): dQ, dK, dV from q, k, v, the
 * forward's output o and LSE, and the output gradient dout. With S = scale q k^T (+ causal
 * mask), P = exp(S - LSE), dP = dout v^T and D = rowsum(dout * o): dS = P * (dP - D),
 * dv = P^T dout, dk = scale dS^T q, dq = scale dS k; with GQA, dk and dv sum over each kv
 * head's query heads. P is recomputed from the LSE. "FlashAttention-3 Deep Dive" (mojostudio.in),
 * the backward-pass sections (recomputation, the D / LSE preprocess, the GQA path);
 * "flash-attention-3" (ai.thesatyajit.com), "Five schedulers" (longest-first causal backward).
 *   q, dout, o, dq: DEVICE bf16 [B, N, H, d]; k, v, dk, dv: DEVICE bf16 [B, N, Hkv, d];
 *   lse: DEVICE fp32 [B, H, N] as attn_fwd wrote it; all 16-byte aligned (lse 4).
 *   workspace: DEVICE, 256-byte aligned, >= attn_bwd_workspace_bytes(B, H, N): D and the base-2
 *   LSE, rows padded to a multiple of 128. Outputs and workspace must not overlap the inputs or
 *   each other. Three kernels on `stream` (preprocess, dK/dV, dQ); no atomics, so the results
 *   are deterministic. INVALID_ARG / UNSUPPORTED as attn_fwd (d == 256 is UNSUPPORTED here);
 *   a bounded wait that gives up is reported by attn_get_status.
 */
size_t attn_bwd_workspace_bytes(int B, int H, int N);
attn_status_t attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                       const void* dout, void* dq, void* dk, void* dv, int B, int H, int Hkv, int N,
                       int d, float scale, int causal, void* workspace, size_t workspace_bytes,
                       cudaStream_t stream);

/* Rows per descale block of the block-scaled e4m3 forward: q in blocks of 128 query positions,
 * k in blocks of 64 key positions, both within one (batch, head). */
#define ATTN_FP8_Q_BLOCK 128
#define ATTN_FP8_K_BLOCK 64

/*
 * attn_fwd_fp8_blockscaled — attn_fwd for e4m3 q, k, v with one descale per block: the score
 * matrix is tiled into 128 x 64 blocks (128 query rows by 64 keys), q carries a descale per
 * 128-row block and k one per 64-row block, so every block of scores has its own scale.
 * "FlashAttention-3 Deep Dive" (mojostudio.in), section 4 "FP8 Block Quantization & Numerical
 * Incoherence Elimination", per-block scaling.
 *   descale_q: DEVICE fp32 [B, H, ceil(N / 128)]; the q value at (b, n, h, :) is
 *              q8 * descale_q[b, h, n / 128].
 *   descale_k: DEVICE fp32 [B, Hkv, ceil(N / 64)]; k at (b, n, g, :) is k8 * descale_k[b, g, n / 64].
 *   descale_v: DEVICE fp32 [B, Hkv]; v at (b, n, g, :) is v8 * descale_v[b, g].
 *   Descales must be positive and finite. attn_quantize_e4m3 writes codes and descales in these
 *   layouts (block_rows 128 for q, 64 for k, N for v). q and k may both be rotated by the same
 *   orthogonal matrix: the scores do not change.
 *   Everything else as attn_fwd with dtype ATTN_DTYPE_FP8_E4M3 (d == 64, 128 or 256).
 */
attn_status_t attn_fwd_fp8_blockscaled(const void* q, const void* k, const void* v, void* o,
                                       float* lse, int B, int H, int Hkv, int N, int d,
                                       float scale, int causal, const float* descale_q,
                                       const float* descale_k, const float* descale_v,
                                       cudaStream_t stream);

/*
 * attn_quantize_e4m3 — bf16 x [B, N, Hx, d] to e4m3 codes x8 [B, N, Hx, d] with one fp32
 * descale per block of block_rows consecutive rows of one (batch, head) (the last block of a
 * head may be shorter): descale = max |x'| / 448 over the block (1 if the block is all zero),
 * x8 = e4m3(x' / descale), rounded to nearest even and saturated to +-448. x' is x, or, when
 * signs is given, x R with R = diag(signs) H_d / sqrt(d), H_d the Sylvester Hadamard matrix:
 * a random orthogonal rotation that spreads outliers across the row. Codes come from the
 * unnormalised product x diag(signs) H_d; the 1/sqrt(d) factor goes into the stored descale.
 * "FlashAttention-3 Deep Dive" (mojostudio.in), section 4: per-block scaling and Hadamard
 * incoherence processing.
 *   x:        DEVICE bf16, 16-byte aligned. Values must be finite.
 *   x8:       DEVICE, 16-byte aligned, B*N*Hx*d bytes; must not overlap x.
 *   descale:  DEVICE fp32 [B, Hx, ceil(N / block_rows)] (attn_quantize_e4m3_descale_count
 *             entries); must not overlap x or x8.
 *   signs:    DEVICE fp32 [d] of +-1 values, or NULL for no rotation. Other values are used as
 *             given (the transform is then not orthogonal).
 *   d in {64, 128, 256}; block_rows >= 1. Blocks of up to 128 rows take one launch; longer
 *   blocks take a memset and three launches on the stream.
 * Asynchronous on stream; allocates nothing. INVALID_ARG for null or misaligned pointers,
 * non-positive sizes or overlapping buffers; UNSUPPORTED for other d or sizes past 32-bit
 * indexing; ATTN_ERR_CUDA if a launch fails.
 */
attn_status_t attn_quantize_e4m3(const void* x, void* x8, float* descale, int B, int N, int Hx,
                                 int d, int block_rows, const float* signs, cudaStream_t stream);

/* Number of descales attn_quantize_e4m3 writes: B * Hx * ceil(N / block_rows) (0 if invalid). */
size_t attn_quantize_e4m3_descale_count(int B, int N, int Hx, int block_rows);

/*
 * attn_fwd_host — the same operation on HOST buffers: copies q, k, v (and the three fp8
 * descales, given here as HOST pointers to one float each) to device buffers owned by the
 * caller (`workspace`, at least attn_fwd_host_workspace_bytes(...) bytes of device memory,
 * 256-byte aligned), runs the forward, and copies o and lse back to host memory.
 * The work is split into up to eight chunks (whole batches when B >= 8, otherwise one batch and a
 * range of KV heads with their query heads), and the first and last chunks are halved when they
 * can be (up to ten in all): their copies overlap no kernel. The upload of one chunk, the kernel
 * of another and the download of a third run concurrently on internal streams (created once per
 * device, never on later calls; the call allocates no memory). The call starts after the work already queued
 * on `stream` and returns after synchronizing `stream`, with o and lse in host memory. Host
 * buffers may be pageable or pinned; only pinned buffers let the copies overlap. Calls on the
 * same device are serialized. Returns as attn_fwd, plus ATTN_ERR_INVALID_ARG for a too-small or
 * misaligned workspace.
 */
attn_status_t attn_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse,
                            int B, int H, int Hkv, int N, int d, float scale, int causal,
                            attn_dtype_t dtype, const float* descale_q, const float* descale_k,
                            const float* descale_v, void* workspace, size_t workspace_bytes,
                            cudaStream_t stream);

/* Device bytes attn_fwd_host needs for one call of this shape (0 for invalid shapes). */
size_t attn_fwd_host_workspace_bytes(int B, int H, int Hkv, int N, int d, attn_dtype_t dtype);

/*
 * attn_fwd_splitkv — split-KV ("flash-decoding") forward for decode-shaped problems: Nq query
 * rows per (batch, head) attend to all Nk keys (no mask: each query sees the whole KV sequence,
 * as a newly generated token sees its cache). The key sequence is cut into
 * min(num_splits, ceil(Nk / 128)) ranges that are processed in parallel, each producing a
 * normalized partial output and its log-sum-exp; a second kernel merges them with
 * LSE = ln sum_s exp(LSE_s), O = sum_s exp(LSE_s - LSE) O_s.
 *   Source: "flash-attention-3" (ai.thesatyajit.com), "What is actually in the box" (split-KV
 *   with a separate combine kernel); "Hopper" tag page (l1-ca0.github.io), section 10 titles
 *   ("Flash-Decoding: Split-KV and the Combine Kernel", 10.2.1 "The combine math") and
 *   section 11 ("PackGQA": query heads of a GQA group are packed into the 128-row tile).
 *
 *   q [B, Nq, H, d], k/v [B, Nk, Hkv, d], o [B, Nq, H, d] bf16, lse [B, H, Nq] fp32: DEVICE
 *   memory, same element types, alignment and descale rules as attn_fwd. H / Hkv must divide
 *   128. 1 <= num_splits <= 128.
 *   workspace: caller-owned DEVICE memory of at least
 *   attn_fwd_splitkv_workspace_bytes(B, H, Nq, d, num_splits) bytes, 256-byte aligned, not
 *   overlapping the other buffers; it holds the partial results and needs no initialization.
 * Asynchronous on `stream`; allocates nothing. Errors as attn_fwd.
 */
attn_status_t attn_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse,
                               int B, int H, int Hkv, int Nq, int Nk, int d, float scale,
                               int num_splits, attn_dtype_t dtype, const float* descale_q,
                               const float* descale_k, const float* descale_v, void* workspace,
                               size_t workspace_bytes, cudaStream_t stream);

/* Device bytes attn_fwd_splitkv needs for its partial results (0 for invalid arguments). */
size_t attn_fwd_splitkv_workspace_bytes(int B, int H, int Nq, int d, int num_splits);

/*
 * attn_splitkv_num_splits — a split count for attn_fwd_splitkv on the current device: the
 * largest S with U * S <= #SMs, where U = B * Hkv * ceil(Nq * H / Hkv / 128) units, clamped to
 * 1 <= S <= min(ceil(Nk / 128), 128). One wave of split units streams K and V near the HBM
 * bandwidth; more splits only add partial results to merge. Host-only; uses 152 SMs when no
 * device can be queried; returns 1 for invalid sizes.
 */
int attn_splitkv_num_splits(int B, int H, int Hkv, int Nq, int Nk, int d);

/* Size of the fixed device scratch used by attn_fwd_splitkv_static (16 MiB). */
#define ATTN_SPLITKV_STATIC_SCRATCH_BYTES (16u * 1024u * 1024u)

/*
 * attn_fwd_splitkv_static — attn_fwd_splitkv for callers that cannot allocate device memory
 * (a plugin whose host framework owns every device allocation, a server that has already
 * committed its memory budget, a latency-critical path that must not risk the device
 * synchronization an allocation can bring). Instead of a caller workspace, the partial results
 * go to a fixed 16 MiB device array that is part of the library (ATTN_SPLITKV_STATIC_SCRATCH_BYTES;
 * every GPU that loads the library holds it until the process exits). The pages have no
 * counterpart to this entry point: it exists for callers of this library.
 *   Arguments, layouts and errors as attn_fwd_splitkv, without workspace arguments. Returns
 *   ATTN_ERR_UNSUPPORTED when attn_fwd_splitkv_workspace_bytes(B, H, Nq, d, S) exceeds
 *   ATTN_SPLITKV_STATIC_SCRATCH_BYTES, where S = min(num_splits, ceil(Nk / 128)) is the number of
 *   splits that run. Allocates nothing, on the device or elsewhere.
 *   The first call in a CUDA context looks up the array's device address (cudaGetSymbolAddress
 *   with the device current) and keeps it for that context; make that first call before any
 *   stream capture. cudaDeviceReset ends the context: the first call after it, in the new
 *   context, looks the address up again (and should again come before any stream capture).
 *   All calls share the one array, and each call overwrites it: calls whose kernels overlap on
 *   the GPU (different streams, or different host threads) race and corrupt each other's results.
 *   Serialize them, e.g. by using one stream. Nothing in the array needs to start at zero: each
 *   call writes every partial result it reads.
 */
attn_status_t attn_fwd_splitkv_static(const void* q, const void* k, const void* v, void* o,
                                      float* lse, int B, int H, int Hkv, int Nq, int Nk, int d,
                                      float scale, int num_splits, attn_dtype_t dtype,
                                      const float* descale_q, const float* descale_k,
                                      const float* descale_v, cudaStream_t stream);

/*
 * attn_get_status — synchronizes `stream`, then returns ATTN_ERR_TIMEOUT if any kernel of this
 * library on the current device gave up a bounded wait since the last attn_clear_status,
 * ATTN_ERR_INVALID_ARG if a varlen forward was handed a plan that does not match it (or that the
 * plan builder marked invalid), ATTN_ERR_CUDA if the synchronization failed, else ATTN_OK.
 */
attn_status_t attn_get_status(cudaStream_t stream);

/*
 * attn_get_status_detail — attn_get_status that also stores the raw device status word in
 * `detail` (may be NULL): 0, 0x40000000 | the code of the wait site that gave up, or 0x2000000C
 * for a rejected varlen plan. 0 is stored when the synchronization fails.
 */
attn_status_t attn_get_status_detail(cudaStream_t stream, uint32_t* detail);

/* attn_clear_status — resets the current device's status word to 0 (synchronous). */
attn_status_t attn_clear_status(void);

/* Human-readable name of a status code (static string; never NULL). */
const char* attn_status_string(attn_status_t s);

/*
 * attn_debug_set — test hook for failure handling. timeout_ns: limit for every bounded wait
 * inside later kernels (0 restores the default of 4 s). skip_load: when nonzero, later launches
 * make CTA 0 skip one K/V tile copy so a wait runs out on purpose; the kernel then unwinds and
 * records ATTN_ERR_TIMEOUT. Process-wide, not thread-safe; for tests only.
 */
void attn_debug_set(unsigned long long timeout_ns, int skip_load);

/* Library version: major * 10000 + minor * 100 + patch. */
int attn_version(void);

#ifdef __cplusplus
}
#endif
#endif /* GB300_ATTN_H */
