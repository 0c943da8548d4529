/*
 * kda.h -- C ABI of the GB300 chunkwise gated delta-rule library (libkda.so).
 *
 * One operator family: DeltaNet (no decay), Gated DeltaNet (scalar per-head
 * log-decay) and Kimi Delta Attention (per-key-channel log-decay), forward
 * and complete backward, over equal-length batches or packed variable-length
 * sequences.
 *
 * Operation (per sequence and head; "Kimi Delta Attention" blog
 * (mainlymatmul.com), section 4, boxed KDA update, in the key-by-value state
 * layout printed at the end of that section):
 *     S~ = diag(exp g_t) S_{t-1};  r_t = beta_t (v_t - S~^T k_t);
 *     S_t = S~ + k_t r_t^T;        o_t = S_t^T (scale q_t)
 * computed chunkwise (chunk length 64) as in "ReWY: Faster Backpropagation
 * for Delta-Rule Attention" (hub.valency.io), sections "The chunk system and
 * conventional WY backward" and Appendix A; the backward pass is the ReWY
 * derivative graph of that paper (Algorithm 1, "State and gate composition",
 * "Matrix intra for vector-gated interactions", "Gram elimination for
 * scalar-gate gradients", "Complete Reverse Execution and Boundaries").
 *
 * Conventions shared by every entry point:
 *  - All tensor pointers are DEVICE pointers, contiguous, row-major, owned by
 *    the caller. The library allocates no device memory for the operator's
 *    tensors or scratch (every buffer is the caller's), frees nothing and does
 *    not synchronise; all work is enqueued on the caller's stream and is
 *    asynchronous. Three things are the library's own: (1) on first use per
 *    host thread and device, one non-blocking side stream and two events,
 *    kept until exit, which carry independent launches beside the caller's
 *    stream and are joined back to it by an event before the call returns;
 *    (2) while tracing is on (kda_profile_begin), CUDA events created on
 *    demand and reused; (3) the static device array of
 *    kda_chunk_fwd_noalloc (see there). kda_device_status and
 *    kda_noalloc_device_status synchronise the stream they are given; they are
 *    diagnostics, not part of the fast path.
 *  - Token tensors use the packed token axis: [B*T, H, X] (equal lengths:
 *    sequence b owns tokens b*T .. b*T+T-1; packed: sequence n owns tokens
 *    cu_seqlens[n] .. cu_seqlens[n+1]-1 and B must be 1).
 *  - States h0, ht, dht, dh0 are fp32 [N, H, K, V] (key-major), N = B, or the
 *    number of packed sequences.
 *  - Arguments are validated before anything is enqueued; on any error
 *    nothing is written and kda_last_error() describes the problem.
 *  - Widths: the chunked calls take any K <= 256 and V <= 4096 (bf16 K, V
 *    multiples of 8 up to 128 and K = V = 256 natively, fp32 K = V = 64 or
 *    128; other widths zero-padded, V above 128 as value blocks, above 256
 *    when K > 128; see kda_problem); the token-by-token call takes K = 64,
 *    128, 160, 192 and 256.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *kda_stream_t;

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = 1,   /* null pointer, bad size, inconsistent fields */
    KDA_ERR_UNSUPPORTED = 2,   /* valid but not built (e.g. K above 256) */
    KDA_ERR_WORKSPACE = 3,     /* workspace or saved buffer too small / misaligned */
    KDA_ERR_CUDA = 4,          /* a launch or runtime call failed */
    KDA_ERR_DEVICE_TIMEOUT = 5 /* a bounded device wait gave up (kda_device_status) */
} kda_status;

/* Element type of q, k, v, beta, o, do, dq, dk, dv, dbeta. */
typedef enum { KDA_BF16 = 0, KDA_FP32 = 1 } kda_dtype;

/* Log-decay kind ("ReWY" paper, Table 1): none (DeltaNet), scalar per token
 * and head (Gated DeltaNet, g is [B*T, H]), per key channel (KDA, g is
 * [B*T, H, K]). */
typedef enum { KDA_GATE_NONE = 0, KDA_GATE_SCALAR = 1, KDA_GATE_CHANNEL = 2 } kda_gate;

typedef struct {
    int B, T, H, K, V;          /* batch, tokens per sequence (total tokens when packed),
                                   heads, key width (1..256), value width (1..4096).
                                   bf16 I/O with K, V <= 128 both multiples of 8 runs
                                   at its own widths (with the in-operator prologue:
                                   K = 64 or 128); K = V = 256, and K = V = 64 or 128
                                   with fp32 I/O, run as they are. Other widths run
                                   zero-padded: bf16 I/O with K <= 128 to 128, fp32 I/O
                                   to 64 (K, V <= 64) or 128, K > 128 to 256 (the value
                                   side too). V above M runs as
                                   ceil(V / M) value blocks, M = 128 (K <= 128) or 256,
                                   each a value head of its own (the delta-rule update
                                   moves every value column of the state independently,
                                   "ReWY" paper, the state recurrence). bf16 I/O at
                                   K <= 128 runs on the tensor cores; K > 128 and fp32
                                   I/O on fp32 CUDA-core kernels. The token-by-token call
                                   needs K = 64, 128, 160, 192 or 256 and V a multiple of
                                   32. */
    int N;                      /* packed sequences (used only when cu_seqlens != NULL) */
    const int32_t *cu_seqlens;  /* device, N+1 non-decreasing token offsets, first 0,
                                   last B*T; NULL for equal-length sequences */
    kda_dtype io;               /* element type of the token tensors */
    kda_gate gate;
    float scale;                /* query scale; <= 0 selects K^-1/2 */
    const void *q, *k;          /* [B*T, H, K] io dtype */
    const void *v;              /* [B*T, H, V] io dtype */
    const void *beta;           /* [B*T, H] io dtype */
    const float *g;             /* natural-log decay, fp32: [B*T, H] (SCALAR) or
                                   [B*T, H, K] (CHANNEL); NULL iff gate == NONE.
                                   Values must satisfy -11 < g <= 0: sub-chunk
                                   factors reach exp(8|g|), which must stay
                                   below the fp32 maximum. */
    const float *h0;            /* [N, H, K, V] fp32 or NULL (zero initial state) */
    int save_policy;            /* 0: backward recomputes the forward (policy R);
                                   1: forward fills `saved` for the backward (policy A) */
    int schedule;               /* backward schedule of the tensor-core path for equal-length
                                   batches: 0 = the library's choice (joint under the save policy
                                   when the pairs fill at most half of the SMs, else one pass);
                                   1 = one reverse-scan pass,
                                   then the consumer; P = 2..8 = P time pieces, the reverse scan
                                   of piece q+1 running beside the consumer of piece q (on a
                                   library-owned second stream); 9 = joint: one cooperative
                                   launch in which the reverse scans run beside the consumer,
                                   which takes each chunk as soon as the scan has written its
                                   state adjoint and sensitivity (save policy, at most one
                                   (sequence, head) pair per SM; else one pass). Results are
                                   identical bitwise for every value; other paths ignore it. */
    /* Optional prologue inside the operator ("GatedDeltaNet-2 (NVlabs) — official spec
     * transcription", §2.0, §3, §4.2); all zero / NULL turns it off. */
    const float *A_log;         /* [H] fp32 or NULL. Non-NULL (needs a gate): g holds the raw gate and
                                   the decay is -exp(A_log) softplus(g + dt_bias) when lower_bound
                                   == 0, else lower_bound sigmoid(exp(A_log) (g + dt_bias)); the
                                   activated decay must meet the bound on g above */
    const float *dt_bias;       /* NULL or fp32 [H, K] (CHANNEL) / [H] (SCALAR); needs A_log */
    float lower_bound;          /* 0 (softplus form) or in [-5, 0) (lower-bound form) */
    int qk_l2norm;              /* 1: q and k are L2-normalised per (token, head) first:
                                   x / sqrt(sum x^2 + l2norm_eps) */
    float l2norm_eps;           /* <= 0 selects 1e-6 */
    /* GatedDeltaNet-2 ("GatedDeltaNet-2 (NVlabs) — official spec transcription", §3): an erase
     * vector per key channel and a write vector per value channel in place of beta,
     *   r_t = write_t .* v_t - S~^T (erase_t .* k_t),  S_t = S~ + k_t r_t^T.
     * Both NULL: the beta rule. Both set: beta is not read (may be NULL); every path takes
     * them (tensor-core, CUDA-core, token-by-token). */
    const void *erase;          /* [B*T, H, K] io dtype */
    const void *write;          /* [B*T, H, V] io dtype */
    /* Grouped value heads: 0 (or H) for one value head per key head. HV = G * H (G > 1): q and
     * k keep H key heads; v, beta, g, erase, write, A_log, dt_bias, h0 and the outputs and
     * gradients of those have HV value heads (read "H" as HV in their shapes above); value
     * head j reads key head j / G, and dq, dk sum over each group. */
    int HV;
} kda_problem;

/* Bytes of device workspace kda_chunk_fwd (for_backward = 0) or kda_chunk_bwd
 * (for_backward = 1) needs for this problem; 0 if the problem is invalid.
 * Only the size fields, io, gate, save_policy, qk_l2norm and whether
 * cu_seqlens, h0, A_log, dt_bias and erase are set are read. The workspace must be 256-byte aligned; its contents need no
 * initialisation and are scratch after the call. */
size_t kda_workspace_size(const kda_problem *p, int for_backward);

/* Bytes of the `saved` buffer used by save_policy 1 (0 for policy 0). */
size_t kda_saved_size(const kda_problem *p);

/* Forward pass. Writes o [B*T, H, V] (io dtype) and, if ht != NULL, the final
 * state of every sequence [N, H, K, V] fp32. With save_policy 1, `saved`
 * (kda_saved_size bytes, 256-byte aligned) receives the chunk intermediates
 * the backward pass reads; it is ignored (may be NULL) under policy 0.
 * Enqueued on `stream`; returns after validation and launch. */
kda_status kda_chunk_fwd(const kda_problem *p, void *o, float *ht, void *saved, void *ws,
                         size_t ws_bytes, kda_stream_t stream);

/* Backward pass of <do, o> + <dht, ht>. Inputs: dout [B*T, H, V] (io dtype),
 * dht [N, H, K, V] fp32 or NULL (zero). With save_policy 1, `saved` must hold
 * what kda_chunk_fwd wrote for the same inputs. Outputs: dq, dk [B*T, H, K],
 * dv [B*T, H, V], dbeta [B*T, H] (io dtype); dg fp32 shaped like g (NULL iff
 * gate == NONE); dh0 [N, H, K, V] fp32 (may be NULL). dq is the gradient with
 * respect to the unscaled q; dg is with respect to the natural-log decay.
 * With the prologue on, dq, dk and dg are with respect to the raw inputs, and
 * dA_log [H] and ddt_bias (shaped like dt_bias) receive the parameters'
 * gradients (each may be NULL; ignored when its parameter is absent). The
 * parameter gradients are sums over tokens formed in a fixed order (no
 * atomics), so repeated calls agree bitwise. With erase/write (GatedDeltaNet-2)
 * dbeta is not written (may be NULL) and derase [B*T, H, K], dwrite
 * [B*T, H, V] (io dtype) receive their gradients; otherwise both are ignored. */
kda_status kda_chunk_bwd(const kda_problem *p, const void *dout, const float *dht,
                         const void *saved, void *dq, void *dk, void *dv, float *dg,
                         void *dbeta, void *derase, void *dwrite, float *dh0, float *dA_log,
                         float *ddt_bias, void *ws, size_t ws_bytes, kda_stream_t stream);

/* Forward pass for callers that cannot allocate device memory: code running
 * inside an allocator's own hooks, processes whose device memory is fully
 * reserved up front by an arena they do not control, or latency-critical
 * paths where an allocation's implicit device synchronisation is not
 * acceptable. The pages have no counterpart to this entry point; it only
 * changes where the forward workspace lives.
 * Same contract as kda_chunk_fwd with save_policy 0, except that the
 * workspace is a library-owned static device array of
 * KDA_NOALLOC_SCRATCH_BYTES (32 MiB) that every device loading the library
 * holds until the process exits. The entry point itself allocates nothing.
 * - Size limit: problems with kda_workspace_size(p, 0) above the array's size
 *   (at K = V = 128 about 450 chunk x head units with bf16 I/O, about 200
 *   with fp32 I/O) are rejected with
 *   KDA_ERR_WORKSPACE before anything is enqueued; save_policy must be 0.
 * - Set-up: the first call on each device, with that device current, looks up
 *   the array's device address (cudaGetSymbolAddress); make that first call
 *   before any stream capture on that device.
 * - Sharing: every call on a device uses the same array, which keeps the last
 *   call's contents; calls whose GPU work overlaps (other streams, other host
 *   threads) race on it and must be serialised by the caller. No word of the
 *   array needs to start at zero: the forward writes all it reads.
 * - Device errors: the error word lives in the array; read it with
 *   kda_noalloc_device_status. */
#define KDA_NOALLOC_SCRATCH_BYTES (32u << 20)
kda_status kda_chunk_fwd_noalloc(const kda_problem *p, void *o, float *ht, kda_stream_t stream);

/* Error word of the last kda_chunk_fwd_noalloc call on the current device, read
 * from the library's static array: synchronises `stream`, then reports as
 * kda_device_status does (KDA_OK when clear, KDA_ERR_DEVICE_TIMEOUT when a
 * bounded wait inside a kernel gave up, KDA_ERR_INVALID_ARG when cu_seqlens
 * was inconsistent). `p` must describe the problem of that call. The pages
 * have no counterpart to this entry point. */
kda_status kda_noalloc_device_status(const kda_problem *p, kda_stream_t stream, int32_t *word);

/* Token-by-token forward for decoding and short prompts ("Kimi Delta
 * Attention" derivation blog, §4 boxed KDA update; the fused recurrent form):
 * the same problem description and tensors as kda_chunk_fwd, save_policy 0.
 * Writes o [B*T, H, V] (io dtype; may be NULL when there are no tokens) and,
 * if ht != NULL, the final states [N, H, K, V] fp32. Needs no workspace: each
 * state is held on chip for the whole call and read and written once, so ht
 * may be the same buffer as p->h0 (the state is updated in place). err is
 * NULL or a device int32 word in which bit 0 is set (atomic OR) when
 * cu_seqlens is inconsistent; such sequences are treated as empty. Any T is
 * accepted, but the tokens of a (sequence, head) are processed one after the
 * other: long prompts belong to kda_chunk_fwd. No backward counterpart.
 * Enqueued on `stream`; returns after validation and launch. */
kda_status kda_recurrent_fwd(const kda_problem *p, void *o, float *ht, int32_t *err, kda_stream_t stream);

/* Synchronises `stream` and reads the device error word a previous call left
 * in `ws` (bit 0: cu_seqlens inconsistent and clamped; bit 1: a bounded wait
 * inside a kernel gave up, so that call's results are not valid). Returns
 * KDA_OK when the word is clear, KDA_ERR_DEVICE_TIMEOUT if bit 1 is set, else
 * KDA_ERR_INVALID_ARG. For diagnostics; the fast path never calls it. */
kda_status kda_device_status(const kda_problem *p, const void *ws, size_t ws_bytes,
                             kda_stream_t stream, int32_t *word);

/* Self-test of the device-timeout path. Enqueues one small kernel (one warp)
 * that waits, with the same bounded mbarrier wait every kernel of the library
 * uses, on a barrier that nothing ever arrives at; after limit_us microseconds
 * (1 .. 1000000) the wait gives up and the kernel sets bit 1 of the device
 * error word in `ws` (the word kda_device_status reads for problem p) and
 * returns. No copy or MMA is in flight during the wait, so the context stays
 * usable; the next kda_chunk_fwd or kda_chunk_bwd on that workspace rewrites
 * the word. `ws` needs at least the chunk-table part of the workspace
 * (kda_workspace_size(p, 0) suffices). The pages have no counterpart to this
 * entry point: it exists so that the timeout reporting can be tested without
 * faulting or hanging a GPU. */
kda_status kda_selftest_device_timeout(const kda_problem *p, void *ws, size_t ws_bytes, unsigned limit_us,
                                       kda_stream_t stream);

/* Message for the last non-OK status returned on the calling thread
 * (thread-local; "" if none). */
const char *kda_last_error(void);

/* Per-kernel device time of the library's own launches (tracing).
 * kda_profile_begin() starts recording a pair of CUDA events around every
 * kernel the library enqueues afterwards (on the stream it is launched on);
 * kda_profile_end() waits for the recorded events, fills up to max_entries
 * records (one per kernel name, in first-launch order) and stops recording.
 * Returns the number of records, or -1 on a CUDA error. Not thread-safe:
 * profile from one host thread. Recording adds one event pair per launch. */
typedef struct {
    char name[40];
    int launches;
    double total_ms;
} kda_kernel_time;

int kda_profile_begin(void);
int kda_profile_end(kda_kernel_time *out, int max_entries);

/* ABI version of this header (bumped on any incompatible change). */
int kda_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
