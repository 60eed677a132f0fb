/*
 * attn.h — C ABI of the GB300 (sm_103a) exact-attention library.
 *
 * Exact scaled-dot-product attention computed tile by tile with an online
 * softmax: per query row the kernels carry a running max m, a denominator l
 * and an output accumulator o, rescaled by exp(m_old - m_new) whenever a new
 * key tile raises the max, so the N x N score and probability matrices never
 * reach device memory ("Explain FlashAttention and why it is IO-aware",
 * "Keep only the state needed for the final weighted average"; "What is
 * FlashAttention?", Steps 2-3). The backward pass recomputes the score and
 * probability tiles from Q, K, V, O and the saved per-row log-sum-exp
 * ("What is FlashAttention?", Step 4; "FlashAttention", "What it does not do").
 *
 * Conventions shared by every entry point:
 *  - Tensors Q, K, V, O (and dO, dQ, dK, dV) are logically [B, H, N, d] with
 *    the last dimension contiguous; the three strides given for (b, h, n) are
 *    in ELEMENTS and may describe any permutation of B/H/N (e.g. BHND or
 *    BNHD). Base pointers and every stride in bytes must be multiples of 16.
 *  - LSE is float32 [B, H, N], contiguous (row-major).
 *  - The caller owns all memory. The library allocates no device memory; the
 *    backward pass uses a caller-provided workspace whose size
 *    attn_bwd_workspace_size() reports.
 *  - Calls are asynchronous on the given stream (a cudaStream_t passed as
 *    void*; NULL is the legacy default stream). Argument errors are found on
 *    the host before anything is launched and are returned directly, with a
 *    message from attn_last_error(). Errors inside a kernel (a bounded wait
 *    that ran out) are recorded in a device error word and reported by the
 *    next attn_status() on that device.
 *  - Launch chaining: the tensor-core kernels and the backward's and decode's
 *    helper kernels are launched with programmatic stream serialization.
 *    Such a kernel may start its on-chip set-up while the kernel before it
 *    on the stream is still finishing. Before it touches device memory it
 *    waits until that kernel has completed and its writes are visible. Stream
 *    order is therefore kept exactly; only the launch gap shrinks.
 *  - Values: Q, K, V and the mask must be finite, except that mask entries
 *    may be -inf ("masked"). NaN or +inf inputs give undefined results (the
 *    pages' row recurrence rejects them up front: "Explain FlashAttention and
 *    why it is IO-aware", "Executable recurrence, with an empty-state
 *    policy"). A query row whose every score is -inf (fully masked) returns
 *    O = 0 and LSE = -inf, and contributes nothing to the gradients (same
 *    section's empty-row policy).
 *  - Empty problems (B, H or N equal to 0) are accepted and do nothing.
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

typedef enum attn_status_t {
    ATTN_OK = 0,
    ATTN_ERR_INVALID = -1,     /* null pointer, negative size, bad flag or stride */
    ATTN_ERR_UNSUPPORTED = -2, /* well-formed but not built: head dim, dtype pairing, size limit */
    ATTN_ERR_ALIGN = -3,       /* a base pointer or byte stride is not a multiple of 16 */
    ATTN_ERR_CUDA = -4,        /* a CUDA runtime or driver call failed */
    ATTN_ERR_TIMEOUT = -5,     /* a kernel's bounded wait ran out (reported by attn_status) */
    ATTN_ERR_WORKSPACE = -6    /* backward workspace missing or smaller than required */
} attn_status_t;

typedef enum attn_dtype_t {
    ATTN_BF16 = 0, /* bfloat16 storage, fp32 accumulation (tcgen05 tensor cores) */
    ATTN_F32 = 1,  /* float32 storage and arithmetic (CUDA cores; forward only)   */
    ATTN_F16 = 2,  /* IEEE half storage, fp32 accumulation (tcgen05 tensor cores);
                      P, dS and O are rounded to half as bf16 rounds them for bf16 */
    ATTN_E4M3 = 3  /* 8-bit E4M3 Q, K, V with per-tensor descale factors; the FP8
                      forward (attn_fwd_fp8) only, whose O is bf16 */
} attn_dtype_t;

/*
 * Forward problem. O = softmax(scale * Q K^T + mask, causal) V and
 * LSE = log(sum_j exp(s_ij)) over the scaled, masked scores of each row
 * ("Explain FlashAttention and why it is IO-aware", "Keep only the state
 * needed for the final weighted average").
 */
typedef struct attn_fwd_params {
    int32_t B, H, N, d;      /* batch, heads, sequence length, head dim: 64 or 128;
                                256 for bf16 / fp16 (forward and attn_bwd) */
    int32_t dtype;           /* attn_dtype_t of Q, K, V, O (and the mask) */
    int32_t causal;          /* 1: key j is masked for query i iff j > i (absolute
                                positions, 0-based; same N for queries and keys) */
    float scale;             /* softmax scale, > 0; 1/sqrt(d) is the usual choice */
    int32_t reserved0;       /* must be 0 */
    const void *q, *k, *v;   /* inputs, device memory */
    void *o;                 /* output, device memory, same dtype as q */
    float *lse;              /* output, device memory, float32 [B, H, N] */
    int64_t q_stride[3];     /* element strides of (b, h, n) */
    int64_t k_stride[3];
    int64_t v_stride[3];
    int64_t o_stride[3];
    const void *mask;        /* optional additive mask, same dtype as q, logically
                                [B, H, N, N] (query row, key column); NULL = none */
    int64_t mask_stride[3];  /* element strides of (b, h, row); 0 broadcasts over
                                that index; the key column is contiguous */
} attn_fwd_params;

/*
 * Backward problem: dQ, dK, dV of sum(dO * O) for the forward described by
 * `fwd`, whose o and lse (as written by attn_fwd) are READ here. Recomputes
 * S and P tile by tile; no gradient flows to the mask. bf16 and fp16 at
 * head dim 64, 128 or 256 (ATTN_F32 returns ATTN_ERR_UNSUPPORTED). At head
 * dim 256 the fp32 dK and dV of one key tile would fill tensor memory, so
 * each key tile is handled by two CTAs, one per half of the head dimension,
 * each recomputing the scores over the whole head dimension: 7/5 of the
 * minimal tensor-core work. ("What is FlashAttention?", "Trade-offs and edge
 * cases": FlashAttention-2 covers head dims up to 256.)
 */
typedef struct attn_bwd_params {
    attn_fwd_params fwd;
    const void *dout;        /* dO, device memory, same dtype as q */
    int64_t do_stride[3];
    void *dq, *dk, *dv;      /* outputs, device memory, same dtype as q */
    int64_t dq_stride[3];
    int64_t dk_stride[3];
    int64_t dv_stride[3];
    void *workspace;         /* device memory, >= attn_bwd_workspace_size(&fwd)
                                bytes, 256-byte aligned; contents need not be
                                initialised and are scratch after the call */
    size_t workspace_bytes;
} attn_bwd_params;

/* Forward pass (every dtype; head dim 256 with bf16 or fp16). */
ATTN_API attn_status_t attn_fwd(const attn_fwd_params *p, void *stream);

/*
 * FP8 forward problem ("What is FlashAttention?", FAQ: FlashAttention-3 has
 * an FP8 forward pass). Q, K and V hold E4M3 codes, one byte per element
 * (sign, 4 exponent bits with bias 7, 3 fraction bits, no infinities), and
 * stand for code value x descale. The result is the attention of those
 * values, as attn_fwd defines it, with the products on the 8-bit tensor
 * cores and P rounded to E4M3 before it multiplies V.
 *  - f.dtype = ATTN_E4M3; f.d = 128 or 256. q, k, v strides count bytes (elements)
 *    and must be multiples of 16. f.o is bf16 [B, H, N, d] (strides in bf16
 *    elements); f.mask, when given, is bf16 as for attn_fwd; f.lse as attn_fwd.
 *  - Accuracy: each probability carries up to 2^-4 relative rounding, so O
 *    differs from the exact attention of the decoded inputs by at most
 *    2^-4 x max|v| per element (plus bf16 output rounding), and typically by
 *    1-3 % in relative L2 norm.
 */
typedef struct attn_fwd_fp8_params {
    attn_fwd_params f;
    float q_descale, k_descale, v_descale;  /* finite and > 0 */
    int32_t reserved1;                      /* must be 0 */
} attn_fwd_fp8_params;

/* FP8 forward pass (tcgen05 kind::f8f6f4). Same conventions and errors as
 * attn_fwd; a 16-bit dtype here, or E4M3 given to attn_fwd, is rejected. */
ATTN_API attn_status_t attn_fwd_fp8(const attn_fwd_fp8_params *p, void *stream);

/* Bytes of workspace attn_bwd needs for this problem (0 for an empty one):
 * per (b, h) and 128-row query tile 1 KiB of fp32 row statistics
 * (-LSE * log2(e) and D = rowsum(dO * O), padded to whole tiles), then the
 * fp32 dQ accumulator [B, H, N, d]. */
ATTN_API size_t attn_bwd_workspace_size(const attn_fwd_params *p);

/* Backward pass: D pre-pass, recompute-and-accumulate kernel, dQ finalize.
 * Head dims 64, 128 and 256 (see attn_bwd_params). */
ATTN_API attn_status_t attn_bwd(const attn_bwd_params *p, void *stream);

/* The same backward pass without a caller workspace: the scratch (row
 * statistics and the fp32 dQ accumulator) lives in a 40 MiB array the
 * library keeps in device memory, so this call allocates nothing. It is for
 * callers that cannot call cudaMalloc or their framework's allocator where
 * they run the backward (inside an allocator callback, in a plug-in whose
 * host owns all memory, under a fixed memory budget). The source pages have
 * no counterpart; it is a convenience of this library.
 *  - Inputs and outputs are passed exactly as for attn_bwd; p->workspace and
 *    p->workspace_bytes are ignored.
 *  - Problems whose attn_bwd_workspace_size() exceeds 40 MiB are rejected
 *    with ATTN_ERR_WORKSPACE before anything is launched.
 *  - Every GPU that loads the library holds the 40 MiB until the process
 *    exits. The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress); make that first call before any stream capture.
 *  - All calls share the one array: calls that overlap on the GPU (other
 *    streams, other threads) race and give wrong gradients. Each call
 *    re-initialises everything it reads, so results do not depend on
 *    earlier calls. Calls queued back to back on one stream do not overlap:
 *    each call's first kernel waits for the previous kernel in the stream.
 *  - The array's address is looked up once per device and kept. The
 *    library must not be used on a device after cudaDeviceReset() (or any
 *    other teardown of its primary context) in the same process: the kept
 *    address would then point at memory the runtime has released. */
ATTN_API attn_status_t attn_bwd_noalloc(const attn_bwd_params *p, void *stream);

/* The backward pass with every gradient reproducible bit for bit: the same
 * inputs give the same dQ, dK and dV on every call and every run on a given
 * GPU model. attn_bwd adds each key tile's share of a dQ row into an fp32
 * accumulator as the tiles finish, so its dQ can differ in the last bits
 * between runs. Here dQ comes from a second tensor-core kernel that keeps a
 * query tile on chip, recomputes the scores and dP against every key tile
 * in order ("What is FlashAttention?", Step 3 loop order, Step 4 recompute)
 * and writes dQ once; dK and dV come from attn_bwd's key-stationary kernel,
 * whose sums over query tiles already run in a fixed order.
 *  - Arguments, workspace and errors exactly as attn_bwd, except that head
 *    dim 256 returns ATTN_ERR_UNSUPPORTED (built for 64 and 128).
 *  - It does about 1.4 times the tensor-core work of attn_bwd (the scores
 *    and dP are computed twice). Results agree with attn_bwd's to rounding. */
ATTN_API attn_status_t attn_bwd_deterministic(const attn_bwd_params *p, void *stream);

/*
 * Decode problem ("FlashAttention", "What it does not do": a decode step reads
 * the whole key/value cache for a few query rows, and what helps is splitting
 * that read across the sequence; "Explain FlashAttention and why it is
 * IO-aware": partial (m, l, o) states merge with the same rescaling as tiles).
 * nq query rows attend to nk >= 1 keys: O = softmax(scale * Q K^T + causal) V
 * per (b, h), with O and LSE as attn_fwd defines them. With causal = 1 the
 * queries are the LAST nq positions: query i sits at position nk - nq + i and
 * sees keys j <= nk - nq + i (a query with none, when nq > nk, gets O = 0 and
 * LSE = -inf). Layouts, alignment and dtypes (bf16 or fp16) as in
 * attn_fwd_params, with separate query and key row counts.
 */
typedef struct attn_decode_params {
    int32_t B, H;
    int32_t nq;              /* query rows per (b, h), 1 .. 128 (from 3 rows up the
                                per-split pass runs on the tensor cores) */
    int32_t nk;              /* keys per (b, h), >= 1 */
    int32_t d;               /* 64 or 128 */
    int32_t dtype;           /* ATTN_BF16 or ATTN_F16 */
    int32_t causal;          /* 0 or 1 (bottom-right aligned, see above) */
    float scale;             /* > 0 */
    const void *q;           /* [B, H, nq, d] */
    const void *k, *v;       /* [B, H, nk, d] */
    void *o;                 /* [B, H, nq, d], dtype of q */
    float *lse;              /* [B, H, nq] fp32, contiguous */
    int64_t q_stride[3], k_stride[3], v_stride[3], o_stride[3]; /* elements, (b, h, row) */
    int32_t num_splits;      /* key ranges per (b, h); 0 = chosen by the library */
    int32_t reserved0;       /* must be 0 */
    void *workspace;         /* >= attn_decode_workspace_size(p) bytes, 256-byte
                                aligned; scratch after the call */
    size_t workspace_bytes;
} attn_decode_params;

/* Bytes of workspace attn_decode needs (the per-split partial states), for
 * the split count it will use (p->num_splits, or its own choice when 0). */
ATTN_API size_t attn_decode_workspace_size(const attn_decode_params *p);

/* Split-KV decode: one kernel computes each split's partial (m, l, o) over
 * its key range, a second merges the splits into O and LSE. Errors as for
 * attn_fwd; nq outside 1 .. 128 returns ATTN_ERR_UNSUPPORTED. */
ATTN_API attn_status_t attn_decode(const attn_decode_params *p, void *stream);

/* Synchronizes `stream`, then reports (and clears) the current device's
 * error word: ATTN_ERR_TIMEOUT if a kernel gave up on a bounded wait since
 * the last call, ATTN_ERR_CUDA for an asynchronous CUDA error, else ATTN_OK. */
ATTN_API attn_status_t attn_status(void *stream);

/* Message for the last non-OK status returned on this host thread ("" if none). */
ATTN_API const char *attn_last_error(void);

/* Upper bound, in nanoseconds, on any single in-kernel wait (mbarrier or
 * pipeline slot) before the kernel records ATTN_ERR_TIMEOUT and returns.
 * Default 2e9 (2 s); values below 1e6 are raised to 1e6. Process-wide. */
ATTN_API void attn_set_wait_timeout_ns(uint64_t ns);

/* Test hook for failure detection: when > 0, the next forward launches on
 * this host thread have their load warp stop after this many key/value
 * tiles, so the consumers' bounded waits run out and report
 * ATTN_ERR_TIMEOUT. 0 (the default) disables it. */
ATTN_API void attn_debug_set_producer_stall(int32_t kv_tiles);

/* Profiling hook: while `events` is non-NULL, every attn_bwd call on this
 * host thread records events[0] before its pre-pass kernel, events[1] after
 * it, events[2] after the recompute kernel and events[3] after the dQ
 * finalize, on the call's stream, so a caller can time each of the three
 * launches with CUDA events. The four cudaEvent_t handles are passed as
 * void* and stay owned by the caller; the array is copied. NULL turns the
 * hook off. */
ATTN_API void attn_debug_set_bwd_events(void *const events[4]);

/* Launch log, for checking on a real system that each call runs as fused
 * kernels ("FlashAttention", "Checking it on a real system": the profiler
 * should show one fused attention kernel, not separate matmul, softmax and
 * matmul launches). attn_debug_launch_count() is the number of kernels this
 * library has launched from the calling host thread since the process
 * started; attn_debug_launch_name(back) is the symbol name of one of the
 * last 16 of them (back = 0 is the most recent), or NULL when `back` is out
 * of that range. The names are the CUDA runtime's (mangled C++ names) and
 * stay valid until the process exits. Every launch is counted once it has
 * been issued without a launch error. */
ATTN_API uint64_t attn_debug_launch_count(void);
ATTN_API const char *attn_debug_launch_name(uint32_t back);

/* Library version, major * 10000 + minor * 100 + patch. */
ATTN_API int32_t attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_ATTN_H */
