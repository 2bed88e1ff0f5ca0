/*
 * attn.h -- C ABI of a fused flash-style attention library for NVIDIA GB300 (sm_103a).
 *
 * What is computed (the plain definition; the kernels reach it without ever forming
 * the S x S score matrix):
 *
 *   s_ij = scale * q_i . k_j                      (query head h reads KV head h / (Hq/Hkv))
 *   allowed(i,j) = j <= i  and  (window <= 0  or  i - j < window)
 *   o_i = sum_j softmax_j(s_ij | allowed) v_j,    lse_i = ln sum_{allowed j} exp(s_ij)
 *
 * with bf16 inputs/outputs, fp32 accumulation and an fp32 log-sum-exp per query row.
 * Passages that define the operation (web pages, by title and section):
 *  - "Gemma4 FFPA attention backend support for accelerating Gemma4-family training"
 *    (NeMo-Automodel discussion 2928): the operator table (fused attention replaces
 *    the MATH path that materialises S x S), "Integration" (head_dim 512 causal full
 *    attention; a 2-D padding mask is served by a varlen path; non-null scale; no
 *    dropout, no softcap) and "Debugging notes" (GQA as repeat-KV).
 *  - "Root cause analysis: Gemma4 sliding-window BF16 cuDNN SDPA NaN on H100"
 *    (NeMo-Automodel issue 3232), "Summary" and "Debug and validation results":
 *    head_dim 256 sliding-window attention whose backward must stay finite in bf16.
 *  - "flex_attention + paged KV + CUDA graphs vs vLLM", "What each option did" and
 *    "Architecture notes": single-token decode over a paged KV cache addressed by a
 *    block table; "What broke correctness": rows with no allowed key must not NaN.
 *
 * Conventions for every entry point:
 *  - All tensor pointers are DEVICE pointers owned by the caller; the library never
 *    allocates, frees or retains them. They must be 16-byte aligned, contiguous, and
 *    live until the work queued on `stream` completes.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).
 *    Calls only enqueue work: they return before the GPU finishes and never
 *    synchronise the device.
 *  - Arguments are checked on the host before anything is launched; on a bad
 *    argument nothing is enqueued and an attn_status code is returned. Nothing
 *    throws across this interface.
 *  - Faults detected on the device (a page id outside the pool, a pipeline wait that
 *    exceeded its time limit) do not trap: the kernel records a flag and finishes,
 *    and attn_get_device_status() reports it.
 *  - Supported shapes: D in {64, 128, 256, 512} for prefill / backward, D in {128, 256} for
 *    decode, D in {64, 128, 256, 512} for the merge; Hq % Hkv == 0, causal = 1. bf16 values
 *    are passed as raw 16-bit patterns.
 */
#ifndef ATTN_GB300_ATTN_H
#define ATTN_GB300_ATTN_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define ATTN_API __attribute__((visibility("default")))
#else
#define ATTN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t attn_bf16; /* raw bf16 bit pattern */

typedef enum attn_status {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = 1,    /* null pointer, negative size, Hq % Hkv != 0, bad scale ... */
    ATTN_ERR_UNSUPPORTED = 2,    /* a legal problem the library has no kernel for (e.g. D = 96) */
    ATTN_ERR_MISALIGNED = 3,     /* a pointer is not 16-byte aligned */
    ATTN_ERR_WORKSPACE = 4,      /* workspace missing or smaller than attn_workspace_size() */
    ATTN_ERR_LAUNCH = 5,         /* the CUDA runtime refused a launch or a tensor map */
    ATTN_ERR_DEVICE_TIMEOUT = 6, /* a kernel pipeline wait gave up (reported by attn_get_device_status) */
    ATTN_ERR_DEVICE_BOUNDS = 7,  /* a device-side index (page id, length) was out of range */
    ATTN_ERR_NO_DEVICE = 8       /* no usable sm_103 device is current */
} attn_status;

/* Operation codes for attn_workspace_size(). */
enum {
    ATTN_OP_FWD = 0,
    ATTN_OP_FWD_VARLEN = 1,
    ATTN_OP_BWD = 2,
    ATTN_OP_BWD_VARLEN = 3,
    ATTN_OP_DECODE_PAGED = 4
};

/*
 * attn_fwd -- causal (optionally sliding-window) attention forward, dense batch.
 *   q   [B, S, Hq,  D] bf16      k, v [B, S, Hkv, D] bf16      (BSHD, contiguous)
 *   o   [B, S, Hq,  D] bf16 out  lse  [B, Hq, S] fp32 out, natural log
 *   scale: finite and > 0 (typically 1/sqrt(D)); causal must be 1; window <= 0 means no
 *   window, otherwise query i sees keys i-window+1 .. i.
 *   workspace: may be NULL (the forward needs none; attn_workspace_size returns 0).
 * Defined by the Gemma4 FFPA page, "Integration" (dense no-mask path) and the
 * sliding-window layers of the issue-3232 page.
 */
ATTN_API int attn_fwd(const attn_bf16* q, const attn_bf16* k, const attn_bf16* v, attn_bf16* o, float* lse, int B, int Hq,
             int Hkv, int S, int D, float scale, int causal, int window, void* workspace, size_t workspace_bytes,
             void* stream);

/*
 * attn_fwd_varlen -- the same forward over packed sequences (the varlen path that
 * replaces a 2-D bool padding mask: Gemma4 FFPA page, "Integration").
 *   q [T, Hq, D], k, v [T, Hkv, D], o [T, Hq, D] bf16; lse [Hq, T] fp32.
 *   cu_seqlens: DEVICE int32 [num_seqs + 1], non-decreasing, cu_seqlens[0] = 0,
 *   cu_seqlens[num_seqs] = total_tokens. Each sequence is its own causal problem.
 *   max_seqlen: an upper bound on every sequence length (sizes the grid without reading
 *   cu_seqlens on the host).
 *   The kernels check every sequence's slice on the device before touching it: a slice
 *   with cu_seqlens[s] < 0, cu_seqlens[s+1] < cu_seqlens[s] (a decreasing prefix sum),
 *   cu_seqlens[s+1] > total_tokens, or a length above max_seqlen is never read or written
 *   (its rows of o and lse keep what they held) and ATTN_ERR_DEVICE_BOUNDS is recorded for
 *   attn_get_device_status(). The other sequences are computed as usual.
 */
ATTN_API int attn_fwd_varlen(const attn_bf16* q, const attn_bf16* k, const attn_bf16* v, attn_bf16* o, float* lse,
                    const int32_t* cu_seqlens, int num_seqs, int total_tokens, int max_seqlen, int Hq, int Hkv, int D,
                    float scale, int causal, int window, void* workspace, size_t workspace_bytes, void* stream);

/*
 * attn_fwd_paged -- chunked prefill over a paged KV cache: each request appends n_b new
 * tokens whose keys and values are already written into its pages, and those n_b queries
 * attend causally to the request's whole cache ("flex_attention + paged KV ..." page,
 * "Architecture notes": keys and values are gathered through the block table).
 *   q [total_q, Hq, D] bf16: the new tokens of all requests, packed; request b owns rows
 *   cu_q[b] .. cu_q[b+1]-1. cu_q: DEVICE int32 [num_reqs + 1], non-decreasing, cu_q[0] = 0,
 *   cu_q[num_reqs] = total_q.
 *   k_cache, v_cache [num_pages, page_size, Hkv, D] bf16; block_table DEVICE int32
 *   [num_reqs, max_pages_per_seq]: page ids of request b in order; seq_lens DEVICE int32
 *   [num_reqs]: L_b, its cached tokens INCLUDING the n_b new ones. New query i of request b
 *   is token L_b - n_b + i and sees keys 0 .. L_b - n_b + i (with window > 0 only the last
 *   `window` of them). n_b = 1 is single-token decode; n_b = L_b is a first prefill.
 *   o [total_q, Hq, D] bf16 out; lse [Hq, total_q] fp32 out (natural log).
 *   max_q_len: an upper bound on every n_b (sizes the grid without reading cu_q on the
 *   host). A request whose cu_q slice leaves [0, total_q) or decreases, with n_b > max_q_len,
 *   n_b > L_b or L_b > max_pages_per_seq * page_size, or a page id outside [0, num_pages), is reported
 *   as ATTN_ERR_DEVICE_BOUNDS by attn_get_device_status() (the bad request's rows are left
 *   unwritten; a bad page id is replaced by page 0). Cache slots past L_b in a request's
 *   last page are never used, whatever they hold.
 *   Supported: D in {64, 128, 256, 512}, page_size = 16, num_reqs <= 65535 / max(1, D / 256).
 *   No workspace.
 *   With num_reqs, total_q or max_q_len zero there is nothing to compute: the call checks
 *   its scalar arguments and returns ATTN_OK, and the pointers may then be NULL.
 */
ATTN_API int attn_fwd_paged(const attn_bf16* q, const attn_bf16* k_cache, const attn_bf16* v_cache,
                            const int32_t* block_table, const int32_t* seq_lens, const int32_t* cu_q, attn_bf16* o,
                            float* lse, int num_reqs, int total_q, int max_q_len, int Hq, int Hkv, int D,
                            int page_size, int max_pages_per_seq, int num_pages, float scale, int causal, int window,
                            void* stream);

/*
 * attn_bwd -- gradient of the forward above with respect to q, k and v, given dO.
 *   Inputs q, k, v, o (the forward's output), lse (the forward's log-sum-exp) and dO in
 *   the forward's layouts; outputs dQ [.., Hq, D], dK, dV [.., Hkv, D] bf16 (dK/dV sum
 *   the contributions of every query head of the KV head's group).
 *   cu_seqlens == NULL: dense [B, S, ...] layout, lse [B, Hq, S].
 *   cu_seqlens != NULL: packed layout with B == 1, S == total tokens, lse [Hq, S], and
 *   num_seqs / max_seqlen as in attn_fwd_varlen. A sequence whose slice fails the device
 *   check described there is reported as ATTN_ERR_DEVICE_BOUNDS: its dK / dV rows are not
 *   written and its dQ rows are zero.
 *   workspace: at least attn_workspace_size(ATTN_OP_BWD[_VARLEN], ...) bytes, 256-byte
 *   aligned; holds an fp32 dQ accumulator and per-row Delta = rowsum(dO * o). Contents on
 *   entry do not matter.
 * The backward recomputes P from lse, never stores it, and must stay finite in bf16
 * (issue-3232 page, "Debug and validation results").
 */
ATTN_API int attn_bwd(const attn_bf16* q, const attn_bf16* k, const attn_bf16* v, const attn_bf16* o, const float* lse,
             const attn_bf16* dO, attn_bf16* dQ, attn_bf16* dK, attn_bf16* dV, int B, int Hq, int Hkv, int S, int D,
             float scale, int causal, int window, const int32_t* cu_seqlens, int num_seqs, int max_seqlen,
             void* workspace, size_t workspace_bytes, void* stream);

/*
 * attn_decode_paged -- one new query token per request over a paged KV cache
 * ("flex_attention + paged KV ..." page, "Architecture notes"), optionally over a sliding
 * window (the head_dim 256 sliding-window layers of the Gemma4 FFPA page at inference).
 *   q [B, Hq, D] bf16; k_cache, v_cache [num_pages, page_size, Hkv, D] bf16;
 *   block_table DEVICE int32 [B, max_pages_per_seq]: page ids of request b in order;
 *   seq_lens DEVICE int32 [B]: cached tokens of request b (the query is token L-1).
 *   window: 0 = the query sees all L cached keys; W > 0 = only keys max(0, L-W) .. L-1 (pages
 *   wholly before the window are not read); W < 0 is rejected.
 *   o [B, Hq, D] bf16 out, lse [B, Hq] fp32 out.
 *   A request with L = 0 gets o = 0 and lse = -inf. Page ids outside [0, num_pages) or
 *   lengths beyond max_pages_per_seq * page_size are not read: the affected tokens are
 *   skipped and ATTN_ERR_DEVICE_BOUNDS is recorded for attn_get_device_status().
 *   Supported: D = 128 with Hq / Hkv in {1, 2, 4, 8}, D = 256 with Hq / Hkv in {1, 2, 4};
 *   page_size = 16, Hkv <= 256, B <= 4096.
 *   workspace: at least attn_workspace_size(ATTN_OP_DECODE_PAGED, B, Hq, Hkv, 0, D, ...) bytes,
 *   256-byte aligned; it holds the split partials of the requests that several CTAs share and
 *   each request's offset into them. Contents on entry do not matter. Calls that share a
 *   workspace must not overlap on the GPU.
 *   Enqueues two kernels on `stream`: the split decode and the merge of its partials, both
 *   launched with programmatic stream serialisation. The merge may become resident while the
 *   decode grid runs and waits on the device for that grid's completion. The decode grid may
 *   start while the kernel enqueued just before it still runs, if that kernel allows dependents
 *   to launch early (the merge of a previous decode call does; a kernel launched without that
 *   attribute, the default, always finishes first): it then reads seq_lens, block_table and the
 *   caches before that kernel has finished, and waits for it only before reading q or writing
 *   the workspace. So a kernel that allows early launch must not write those three inputs of
 *   the decode call that follows it. In particular the o / lse of one decode call may be the q
 *   of the next, but not its caches, block_table or seq_lens.
 */
ATTN_API int attn_decode_paged(const attn_bf16* q, const attn_bf16* k_cache, const attn_bf16* v_cache,
                      const int32_t* block_table, const int32_t* seq_lens, attn_bf16* o, float* lse, int B, int Hq,
                      int Hkv, int D, int page_size, int max_pages_per_seq, int num_pages, float scale, int window,
                      void* workspace, size_t workspace_bytes, void* stream);

/*
 * attn_decode_paged_noalloc -- attn_decode_paged for callers that cannot allocate device
 * memory (no counterpart on the pages; added for integrators). Some callers cannot call
 * cudaMalloc on their decode path: a plug-in inside a host application that owns the
 * whole device-memory budget through its own pool, or a latency-critical token loop where
 * cudaMalloc's implicit device synchronisation would stall other streams. This variant
 * takes no workspace: the kernel's scratch comes from a 16 MiB buffer compiled into the
 * library (attn_decode_paged_noalloc_max_bytes()), which every GPU that loads the library
 * keeps until the process exits. It allocates nothing and calls no allocating routine.
 *   Arguments, layouts and results are those of attn_decode_paged.
 *   Limit: attn_workspace_size(ATTN_OP_DECODE_PAGED, B, Hq, Hkv, 0, D, 0, max_pages) must
 *   not exceed attn_decode_paged_noalloc_max_bytes() (e.g. Hq = 32 allows B up to 240);
 *   larger problems are rejected with ATTN_ERR_WORKSPACE before anything is enqueued.
 *   The first call made while a given device is current looks up the buffer's device
 *   address (cudaGetSymbolAddress) for that device and caches it for the life of the
 *   process; make that first call before any stream capture on the device. The cached
 *   address does not survive cudaDeviceReset(): after a reset of a device, do not call this
 *   entry point on it again in the same process.
 *   All calls on a device share the one buffer, and it keeps the previous call's contents.
 *   Nothing in it needs to start at zero: every call writes all of it that it reads.
 *   Calls whose execution overlaps on the GPU (different streams without ordering) race
 *   on the buffer and give wrong results: order them.
 */
ATTN_API int attn_decode_paged_noalloc(const attn_bf16* q, const attn_bf16* k_cache, const attn_bf16* v_cache,
                                       const int32_t* block_table, const int32_t* seq_lens, attn_bf16* o, float* lse,
                                       int B, int Hq, int Hkv, int D, int page_size, int max_pages_per_seq,
                                       int num_pages, float scale, int window, void* stream);

/* attn_decode_paged_noalloc_max_bytes -- size of the built-in decode scratch buffer (bytes). */
ATTN_API size_t attn_decode_paged_noalloc_max_bytes(void);

/*
 * attn_merge_lse -- combine attention results computed over disjoint sets of keys into the
 * attention over all of them: the combining step of context-parallel ring attention, where each
 * ring chunk of keys is attended separately ("Gemma4 FFPA attention backend support ..." page,
 * "Integration"). Part p holds o_p, normalised over its own keys, and lse_p (natural log of the
 * sum of exp(scale * q.k) over them), as every forward of this library returns them. Per row:
 *   lse = ln sum_p exp(lse_p),   o = sum_p exp(lse_p - lse) * o_p   (fp32, o rounded to bf16)
 * A part with lse_p = -inf (no allowed key) contributes nothing, whatever its o_p holds; a row
 * with no key in any part gets o = 0, lse = -inf. lse values must be finite or -inf.
 *   o_parts [num_parts, B, S, H, D] bf16 and lse_parts [num_parts, B, H, S] fp32: the parts
 *   stacked in the forward's layouts (packed [T, H, D] / [H, T] results: B = 1, S = T).
 *   o [B, S, H, D] bf16 out, lse [B, H, S] fp32 out. The outputs may be part 0's own buffers
 *   (o == o_parts and lse == lse_parts: a running merge in place); any other overlap between
 *   inputs and outputs is not allowed.
 *   Supported: D in {64, 128, 256, 512}, 1 <= num_parts <= 64. o_parts and o 16-byte aligned.
 *   With B, S or H zero there is nothing to do and the pointers may be NULL. No workspace.
 */
ATTN_API int attn_merge_lse(const attn_bf16* o_parts, const float* lse_parts, attn_bf16* o, float* lse, int num_parts,
                            int B, int S, int H, int D, void* stream);

/*
 * attn_workspace_size -- bytes of workspace an operation needs (0 if none).
 *   For ATTN_OP_BWD: B, Hq, S, D; for ATTN_OP_BWD_VARLEN pass B = 1 and S = total tokens.
 *   For ATTN_OP_DECODE_PAGED: B, Hq, Hkv, D. Unused arguments are ignored. Returns 0 for an
 *   unknown op, and for a decode problem no decode kernel takes (D not 128 / 256, Hq not a
 *   supported multiple of Hkv), whose call is rejected anyway. Pure host arithmetic; needs no
 *   GPU.
 */
ATTN_API size_t attn_workspace_size(int op, int B, int Hq, int Hkv, int S, int D, int num_seqs, int max_pages_per_seq);

/*
 * attn_get_device_status -- synchronise `stream`, then read and clear the device fault
 * flags raised by kernels of this library on the current device. Returns ATTN_OK,
 * ATTN_ERR_DEVICE_TIMEOUT, ATTN_ERR_DEVICE_BOUNDS, or ATTN_ERR_LAUNCH if the stream
 * itself reports a CUDA error.
 */
ATTN_API int attn_get_device_status(void* stream);

/*
 * attn_selftest_wait_timeout -- exercise the failure-reporting path of the kernels' pipeline
 * waits (no counterpart on the pages). Enqueues on `stream` one small kernel whose single
 * thread waits on an mbarrier phase that nothing completes, with the same bounded wait the
 * attention kernels use but a limit of `limit_ms` milliseconds (1..10000). The wait gives up,
 * the kernel records ATTN_ERR_DEVICE_TIMEOUT in the device status and returns normally: no
 * fault, no hang, and the context stays usable. Returns ATTN_OK once enqueued,
 * ATTN_ERR_INVALID_ARG for a limit out of range; read the outcome with
 * attn_get_device_status().
 */
ATTN_API int attn_selftest_wait_timeout(int limit_ms, void* stream);

/* attn_status_string -- a static, human-readable name for a status code. */
ATTN_API const char* attn_status_string(int status);

/* attn_version -- library version as MAJOR * 10000 + MINOR * 100 + PATCH. */
ATTN_API int attn_version(void);

/*
 * Observability (no counterpart on the pages; used by the benchmark):
 * attn_launch_count -- number of kernel launches this library has issued in this process.
 * attn_profile_start -- from now on, bracket every kernel launch with a pair of CUDA events
 *   on the launching stream (discards earlier records). Do not enable while capturing a
 *   CUDA graph.
 * attn_profile_stop -- stop recording, wait for the recorded events, and write one line per
 *   kernel, "name launches total_ms\n", into buf (NUL-terminated, truncated to buf_bytes).
 *   Returns the number of distinct kernels, or -ATTN_ERR_LAUNCH if an event failed.
 */
ATTN_API unsigned long long attn_launch_count(void);
ATTN_API int attn_profile_start(void);
ATTN_API int attn_profile_stop(char* buf, size_t buf_bytes);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_ATTN_H */
