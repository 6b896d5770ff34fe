/*
 * cpdr.h -- C ABI of the segmented ("True CP") gated delta-rule forward for
 * GB300 (sm_103a).
 *
 * The operation is the one described in the article
 *   "flash-linear-attention 上下文并行CP从 CP2TP、Ring CP 到 True CP 的设计取舍
 *    与源码实现"                                     (cited below as [FLA-CP])
 * run on ONE GPU with the sequence cut into R contiguous segments that play
 * the role of context-parallel ranks:
 *
 *   per token      S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
 *                  o_t = scale * S_t^T q_t                      alpha_t = exp(g_t)
 *   preprocess     every segment j computes, from a zero state, the state of
 *                  its trailing fragment S_ext,j (dk x dv) and the product of
 *                  that fragment's transfer matrices M_j (dk x dk), in the
 *                  chunk (WY) form with 64-token chunks    ([FLA-CP] §2.1-§2.3)
 *   merge          S_init,r = sum over predecessors: S <- M_j S + S_ext,j
 *                                                          ([FLA-CP] §2.1, §5.2)
 *   fwd            every fragment restarts from S_init (its segment's first
 *                  fragment, when it continues a sequence) or zero, and emits
 *                  o and the final state of sequences ending in it
 *                                                          ([FLA-CP] §4, §5.2)
 *
 * Conventions shared by every entry point
 * ----------------------------------------
 * Layout.  q: [B, T, Hq, dk]; k: [B, T, H, dk]; v: [B, T, H, dv];
 *          o: [B, T, Hq, dv] (Hq == H unless desc.Hq asks for grouped query
 *          heads); beta: [B, T, H];
 *          gate: [B, T, H] (scalar, GDN) or [B, T, H, dk] (per key dim, KDA),
 *          all contiguous, row-major.  Packed variable-length batches use
 *          B == 1 and global cu_seqlens ([FLA-CP] §3.1, §4 NOTE).
 *          S_ext, S_init: [R, B, H, dk, dv] fp32; M: [R, B, H, dk, dk] fp32
 *          (entry (r, b, h) belongs to segment r of row b; the layout of the
 *          gathered buffer of [FLA-CP] §2.4 with world_size = R);
 *          final_state: [N, H, dk, dv] fp32 ([N, HV, K, V] of the KDA
 *          initial_state description in hyper-parallel issue #7).  With
 *          CPDR_FLAG_STATE_V_FIRST the dk x dv states are [.., dv, dk]; with
 *          CPDR_FLAG_LAYOUT_ZIGZAG the token axis is in zigzag order and the
 *          segment axis has 2R entries.
 * Types.   q, k, v, beta, o share the input dtype (fp32 or bf16); gates are
 *          fp32 natural-log gates g = log(alpha).  Arithmetic is fp32 or
 *          bf16 tensor-core products with fp32 accumulation; the M chain is
 *          kept at fp32 accuracy ([FLA-CP] §2.2).
 * Memory.  Every tensor argument is a DEVICE pointer owned by the caller, and
 *          must be 16-byte aligned.  The library owns only the cpdr_ctx
 *          (host tables plus small device metadata allocated at create,
 *          and two copy streams and twelve events for cpdr_forward_host).
 *          No call below allocates device memory.
 * Streams. `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *          stream).  Calls enqueue work and return; they never synchronise.
 *          Every stage runs on `stream` (cpdr_forward_host also uses the
 *          context's copy streams, ordered against `stream` by events); a
 *          context must not be used from two host threads at once.
 * Errors.  Every call validates its arguments on the host before any
 *          launch and returns a cpdr_status; on failure nothing is launched
 *          and cpdr_last_error() gives a message (thread-local).  Launch
 *          failures come back as CPDR_ERR_CUDA.
 */
#ifndef CPDR_H_
#define CPDR_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    CPDR_OK = 0,
    CPDR_ERR_INVALID = 1,      /* bad shapes, cut rule violated, null/misaligned pointers */
    CPDR_ERR_UNSUPPORTED = 2,  /* valid but not implemented (e.g. dk != dv, d not in {64,128}) */
    CPDR_ERR_CUDA = 3,         /* a CUDA runtime call or kernel launch failed */
    CPDR_ERR_WORKSPACE = 4,    /* a caller-provided buffer is too small */
    CPDR_ERR_TIMEOUT = 5       /* a bounded device-side wait gave up (see cpdr_check_device_status) */
} cpdr_status;

/* desc.flags */
#define CPDR_FLAG_HOST_ONLY   (1u << 0)  /* plan only: no device tables; launch calls are rejected */
#define CPDR_FLAG_FORCE_SIMT  (1u << 1)  /* use the fp32 CUDA-core kernels even where tensor cores apply */
/* Zigzag token layout ([FLA-CP] §3.2).  Each row (or the packed batch) is cut
 * into 2R equal parts; virtual rank r holds part r followed by part 2R-1-r, and
 * the tensors q, k, v, beta, gate and o hold the R ranks' [front; back] inputs
 * side by side, rank 0 first (for R = 2: parts 0, 3, 1, 2 in memory).
 * cu_seqlens stays in sequence order.  Every part is a segment of its own, so
 * the exchange buffers have 2R entries, indexed by part in sequence order, and
 * the cut rule becomes "tokens >= 2R and divisible by 2R". */
#define CPDR_FLAG_LAYOUT_ZIGZAG (1u << 2)
/* state_v_first ([FLA-CP] §5.1; [N, HV, V, K] of hyper-parallel issue #7):
 * every dk x dv state buffer -- S_ext, S_init and final_state -- is stored
 * transposed, [.., dv, dk].  M keeps its [.., dk, dk] layout. */
#define CPDR_FLAG_STATE_V_FIRST (1u << 3)

/* desc.gate_kind */
#define CPDR_GATE_SCALAR  0   /* GDN: g [B, T, H] */
#define CPDR_GATE_PER_DIM 1   /* KDA: gk [B, T, H, dk] */

/* desc.in_dtype */
#define CPDR_DTYPE_F32  0
#define CPDR_DTYPE_BF16 1

typedef struct {
    int32_t B, H, dk, dv;   /* batch rows, heads, key dim, value dim */
    int32_t R;              /* virtual context ranks: R contiguous segments per row (or 2R
                               zigzag pieces, see CPDR_FLAG_LAYOUT_ZIGZAG) */
    int32_t num_seqs;       /* N: sequences (== B without cu_seqlens) */
    int64_t T;              /* tokens per row, or total tokens when packed */
    const int64_t *cu_seqlens_host; /* NULL: B rows of T tokens; else N+1 global offsets
                                       (host memory, read during create only), B == 1 */
    int32_t gate_kind;      /* CPDR_GATE_* */
    int32_t in_dtype;       /* CPDR_DTYPE_* */
    uint32_t flags;         /* CPDR_FLAG_* */
    float scale;            /* output scale */
    int32_t Hq;             /* query heads of q and o (GQA, [FLA-CP] §5.1): 0 or H for none,
                               else a multiple G*H; q head hq reads the state of head hq / G,
                               while k, v, beta, gate and every state keep H heads */
    int32_t conv_width;     /* causal conv1d kernel size W for cpdr_conv1d_fwd (the
                               conv1d_kernel_size of [FLA-CP] §3.1-§3.2): 0 = no conv path,
                               else 1..8 */
} cpdr_desc;

typedef struct cpdr_ctx cpdr_ctx;

/* One local fragment: the intersection of a segment with a sequence. */
typedef struct {
    int64_t tok0;    /* first token on the flattened [B*T] token axis, where it is in
                        memory (zigzag layout: its memory position, not its sequence position) */
    int32_t len;     /* tokens (>= 1) */
    int32_t seg;     /* segment buffer index r*B + b */
    int32_t seq;     /* sequence index */
    int32_t flags;   /* CPDR_FRAG_* */
} cpdr_fragment;

#define CPDR_FRAG_CONT_PREV 1   /* continues a sequence from segment r-1: starts from S_init[seg] */
#define CPDR_FRAG_CONT_NEXT 2   /* continues into segment r+1: pre-processed into S_ext/M[seg] */
#define CPDR_FRAG_ENDS_SEQ  4   /* the sequence ends here: final_state[seq] is written */

/*
 * Build the partition plan ([FLA-CP] §3.2-§3.3: contiguous layout, the cut
 * rule "tokens >= R and divisible by R" per row, searchsorted-style
 * intersection of the global cu_seqlens with each segment) and upload its
 * small device tables (unless CPDR_FLAG_HOST_ONLY).  The plan is built once
 * and reused, like the memoised context of [FLA-CP] §3.3.
 * Errors: CPDR_ERR_INVALID (cut rule, non-monotone cu_seqlens, B != 1 with
 * cu_seqlens, non-positive sizes), CPDR_ERR_UNSUPPORTED (dk != dv or
 * d not in {64, 128}), CPDR_ERR_CUDA (table upload).  *out is NULL on error.
 */
cpdr_status cpdr_ctx_create(const cpdr_desc *desc, cpdr_ctx **out);

/* Free the context and its device tables.  NULL is accepted. */
void cpdr_ctx_destroy(cpdr_ctx *ctx);

/* Byte sizes of the caller-owned exchange buffers S_ext, M, S_init and of
 * final_state.  Any pointer may be NULL. */
cpdr_status cpdr_buffer_sizes(const cpdr_ctx *ctx, size_t *sext_bytes, size_t *m_bytes,
                              size_t *sinit_bytes, size_t *final_bytes);

/* Plan introspection (host memory): number of fragments, and a copy of the
 * fragment table into out[0 .. min(cap, n)). */
cpdr_status cpdr_plan_num_fragments(const cpdr_ctx *ctx, int32_t *n);
cpdr_status cpdr_plan_fragments(const cpdr_ctx *ctx, cpdr_fragment *out, int32_t cap);

/* Plan counters (host memory): out[0] fragments, [1] pre-processed
 * fragments, [2] merge chains, [3] segments with zeroed S_ext/M, [4]
 * segments with zeroed S_init, [5] empty sequences, [6] kernel launches per
 * preprocess+merge+fwd step, [7] 1 if the tensor-core kernels are selected. */
cpdr_status cpdr_plan_counts(const cpdr_ctx *ctx, int32_t out[8]);

/*
 * WY build ([FLA-CP] §2.2 and the recompute_w_u step of its §4 Code Flow):
 * for every 64-token chunk of every fragment and every head,
 *     A_ij = beta_i exp(G_i - G_j) k_i . k_j  (j < i),   T = (I + A)^-1,
 * with G the in-chunk cumulative log gate, and the tiles W and U are built
 * from:  T' = T diag(beta)  (U = T' V)  and  T'' = T diag(beta gamma)
 * (W = T'' K, gamma_j = exp(G_j)).  Each (chunk, head) gets three 64 x 64
 * bf16 tiles -- T', T'' rounded (hi) and T'' - hi rounded (lo) -- stored as
 * 8 KiB 128-byte-swizzled images, in the chunk order of the plan's fragment
 * table, heads innermost.  The chunk recurrences of cpdr_preprocess and
 * cpdr_fwd read them (the triangular solve is independent across chunks, so
 * it runs here once, fully parallel, instead of inside every chain).
 * cpdr_wy_bytes() gives the workspace size: 24 KiB per (chunk, head) on the
 * tensor-core path (bf16, dk = dv = 128, scalar gate), 0 otherwise (then
 * this call does nothing and `wy` may be NULL).
 * Per-dim gate (KDA) on the tensor-core path: the gate cannot be applied
 * inside the chunk recurrence as a scalar, so this step also pre-gates the
 * operands, as [FLA-CP] §2.3 does at the WY stage (kg = k 2^(g_last - g),
 * qg = q 2^g): per (chunk, head) it writes, after the three tiles above
 * (built with gamma = 1), the per-dim chunk decay 2^(G_C), the bf16 tiles
 * k 2^G (hi, lo), k 2^(G_C - G) (hi, lo), q 2^G and the masked intra-chunk
 * product (Q K^T ⊙ Lambda) -- 113 KiB per (chunk, head).  With grouped
 * query heads (Hq = G H) the unit holds q 2^G and the product of its state's
 * first query head; those of query heads 1 .. G-1 (24 KiB each) follow all
 * units, [chunk][head][G - 1].
 * In: q (device; read only for the per-dim gate, else may be NULL), k,
 * beta, gate (device).  Out: wy (device, caller-owned).
 */
cpdr_status cpdr_wy_bytes(const cpdr_ctx *ctx, size_t *bytes);
cpdr_status cpdr_wy_build(const cpdr_ctx *ctx, const void *q, const void *k, const void *beta,
                          const float *gate, void *wy, void *stream);

/*
 * Pre-process ([FLA-CP] §2.1-§2.3, pre_process_fwd in its Code Flow of §4):
 * for every segment whose trailing fragment continues into the next
 * segment, S_ext = state of that fragment from zero, M = chained transfer
 * matrix  M <- (Diag(gamma^C) - (Gamma ⊙ K)^T W) M  over its 64-token
 * chunks.  Entries of segments with no continuing fragment are zeroed.
 * In: k, v, beta, gate (device); wy: the tiles cpdr_wy_build wrote for the
 * same k, beta and gate (NULL when cpdr_wy_bytes() is 0).  Out: S_ext, M
 * (device, sizes from cpdr_buffer_sizes).
 */
cpdr_status cpdr_preprocess(const cpdr_ctx *ctx, const void *k, const void *v, const void *beta,
                            const float *gate, const void *wy, float *S_ext, float *M, void *stream);

/*
 * Merge ([FLA-CP] §2.1; ownership rule of §5.2): for every segment r whose
 * first fragment continues a sequence begun in segment r - n_pre,
 *     S = 0;  for j = r - n_pre .. r - 1:  S <- M_j S + S_ext,j
 * and S_init[r] = S; all other entries are zeroed.  Evaluated as one
 * sequential scan per sequence (equal in exact arithmetic).  Precision: on
 * the tensor-core path (bf16 inputs, d = 128) each product M_j S runs on the
 * tensor cores with M_j and S split into bf16 hi/lo pairs and fp32
 * accumulation (about 2^-16 relative per step); otherwise all fp32.
 * In: S_ext, M (device, as cpdr_preprocess wrote them).  Out: S_init
 * (device).  Errors: CPDR_ERR_INVALID, CPDR_ERR_CUDA.
 */
cpdr_status cpdr_merge(const cpdr_ctx *ctx, const float *S_ext, const float *M, float *S_init,
                       void *stream);

/*
 * Forward ([FLA-CP] §4, chunk_gated_delta_rule_fwd_h plus the output step):
 * every fragment runs the 64-token chunk recurrence from S_init[seg] (first
 * fragment continuing a sequence) or zero, writes o = scale * S_t^T q_t per
 * token and, when its sequence ends there, final_state[seq].
 * wy: as for cpdr_preprocess.  final_state may be NULL.
 */
cpdr_status cpdr_fwd(const cpdr_ctx *ctx, const void *q, const void *k, const void *v,
                     const void *beta, const float *gate, const void *wy, const float *S_init, void *o,
                     float *final_state, void *stream);

/*
 * Causal depthwise conv1d over the token axis, the layer step before the
 * delta rule, on the context's segments ([FLA-CP] §2.4: the conv sees only
 * the W - 1 tokens before each token, so a rank takes the tail of the
 * previous rank's tokens; §3.2-§3.3: conv1d_kernel_size, pre_num_conv_tokens).
 * Per channel c and token t of a sequence (positions before the sequence
 * start read as zero):
 *     y[t, c] = act( bias[c] + sum_{i=0}^{W-1} weight[c, i] * x[t - (W-1) + i, c] )
 * act = identity (activation 0) or SiLU, z * sigmoid(z) (activation 1).
 * On one device the previous segment's tail is read where it lies in memory
 * (in the zigzag layout, another rank's part), so no exchange buffer exists.
 * Layout: x, y [B, T, channels] in the context's token order and input dtype
 * (fp32 or bf16), contiguous; weight [channels, W] fp32; bias [channels] fp32
 * or NULL.  W = desc.conv_width (> 0).  channels % 8 == 0, 1 <= channels.
 * Arithmetic in fp32, y rounded once.  y must not overlap x.
 * Errors: CPDR_ERR_INVALID (context without a conv width, bad channels or
 * activation, null or misaligned pointers), CPDR_ERR_CUDA.
 */
cpdr_status cpdr_conv1d_fwd(const cpdr_ctx *ctx, const void *x, const float *weight, const float *bias,
                            int32_t channels, int32_t activation, void *y, void *stream);

/*
 * Backward ([FLA-CP] §2.2 and §4 split it into a pre-process, the merge run
 * in reverse with the transposed transfer matrices, and state-gradient
 * chains): the gradients of  sum_t <do_t, o_t> + sum_n <dht_n, final_state_n>
 * with respect to q, k, v, beta and the gate, for the same inputs the
 * forward ran on.
 *   1. each segment's first fragment that continues a sequence runs the
 *      reverse chain from its local end gradient (dht if its sequence ends
 *      there, else 0) and keeps the state gradient at its start, dS_ext;
 *   2. per sequence crossing cuts:  G = dS_ext[r1];
 *      for j = r1-1 .. r0+1:  G <- M_j^T G + dS_ext[j]  (the gradient at the
 *      end of every continuing fragment);
 *   3. every fragment runs the reverse chain from that end gradient (or dht,
 *      or 0) and writes the input gradients.
 * For bf16 inputs and dk = dv = 128 (either gate) the chains run in chunk form on the tensor
 * cores: the forward is recomputed with every chunk's starting state and
 * Delta kept, the state-gradient chain runs chunk by chunk in reverse
 * (tcgen05), the reverse merge on the tensor cores, and a parallel kernel
 * forms the input gradients of every (chunk, head) (for the per-dim gate
 * with its factors folded into the operands); the workspace then holds the
 * WY tiles (the per-dim gate's units), the fp32 inverse T and four fp32
 * tensors per (chunk, head) (about 216 KiB each).  Otherwise the reverse
 * chain is the per-token chain rule, on CUDA cores in fp32, with the
 * forward states recomputed from S_init per token.  With grouped query
 * heads (Hq = G H) each state's chain takes the G query heads that read it
 * ([FLA-CP] §5.1): its state gradient collects scale q do^T of every one of
 * them, and each gets its own dq (on the tensor cores the chunk-form
 * state-gradient chain, linear in those terms, runs once per query head and
 * sums, and the input-gradient kernel makes a pass per query head).
 * In (device): q, k, v, beta, gate and do ([B, T, Hq, dv], the input dtype)
 * as for cpdr_fwd; dht [N, H, dk, dv] fp32 (with CPDR_FLAG_STATE_V_FIRST
 * [N, H, dv, dk]) or NULL (zero); S_init and M as cpdr_merge and
 * cpdr_preprocess left them for these inputs.  Out (device, fp32, written
 * here): dq [B, T, Hq, dk], dk [B, T, H, dk], dv [B, T, H, dv], dbeta
 * [B, T, H], dgate (the gate's shape).  workspace: device memory of
 * cpdr_bwd_workspace_bytes() bytes, 256-byte aligned.
 * Errors: CPDR_ERR_UNSUPPORTED when the G query heads' rows of one chunk do
 * not fit the CUDA-core chain's shared memory (at d = 128: G above 8 for
 * bf16 with the scalar gate, 6 with the per-dim gate; 4 and 3 for fp32);
 * CPDR_ERR_WORKSPACE; CPDR_ERR_INVALID; CPDR_ERR_CUDA.
 */
cpdr_status cpdr_bwd_workspace_bytes(const cpdr_ctx *ctx, size_t *bytes);
cpdr_status cpdr_bwd(const cpdr_ctx *ctx, const void *q, const void *k, const void *v, const void *beta,
                     const float *gate, const void *dout, const float *dht, const float *S_init, const float *M,
                     float *dq, float *dk, float *dv, float *dbeta, float *dgate, void *workspace,
                     size_t workspace_bytes, void *stream);

/* pre_num_conv_tokens ([FLA-CP] §3.3) per segment, host memory: how many of
 * the W - 1 tokens before segment s's start belong to its first sequence
 * (0 when the segment starts a sequence), out[0 .. min(cap, nseg)). */
cpdr_status cpdr_plan_conv_tokens(const cpdr_ctx *ctx, int32_t *out, int32_t cap);

/*
 * Whole path from HOST memory: copies q, k, v, beta, gate into the
 * caller-provided device workspace, runs the WY build, preprocess, merge and fwd on
 * `stream`, and copies o and final_state back (host pointers; use pinned
 * memory for asynchronous copies).  Returns after enqueuing; the caller
 * synchronises the stream before reading o.  The workspace must hold
 * cpdr_host_workspace_bytes() bytes (256-byte aligned device memory).
 * The host-to-device copies run on the context's copy stream, ordered after
 * all work enqueued on `stream` before the call, in the order the stages
 * need them (k, beta, gate, then v, then q in four groups of consecutive
 * tokens); each stage waits on `stream` for its own inputs only, the
 * forward runs group by group, and each group's o is copied back on the
 * context's output stream while the next group runs; `stream` waits for
 * the last copy before anything later on it.
 */
cpdr_status cpdr_host_workspace_bytes(const cpdr_ctx *ctx, size_t *bytes);
cpdr_status cpdr_forward_host(const cpdr_ctx *ctx, const void *q, const void *k, const void *v,
                              const void *beta, const float *gate, void *o, float *final_state,
                              void *device_workspace, size_t workspace_bytes, void *stream);

/*
 * Allocation-free whole path (no counterpart in the article: it is an
 * interface for callers that cannot allocate device memory, e.g. code inside
 * a runtime that owns all device memory through its own pool or static
 * memory plan).  Runs the WY build, preprocess, merge and fwd like the calls
 * above, but keeps everything except the caller's inputs and outputs -- the
 * WY tiles, the exchange buffers S_ext, M, S_init, the plan tables and the
 * status word of the bounded waits -- in one file-scope device array of
 * 32 MiB per device
 * (held by every GPU that loads the library until the process exits).  It
 * calls no cudaMalloc, cudaFree or other allocating routine, and accepts a
 * context created with CPDR_FLAG_HOST_ONLY.
 * In: q, k, v, beta, gate (device).  Out: o, final_state (device; final_state
 * may be NULL).  Errors: CPDR_ERR_WORKSPACE when the problem needs more than
 * the array holds (R*B*H*dk*(2*dv + dk)*4 bytes of exchange buffers, the WY
 * tiles of cpdr_wy_bytes() and the plan tables), CPDR_ERR_INVALID / CPDR_ERR_CUDA as for the other calls.
 * Set-up: the first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture.  Every call shares the one array and overwrites
 * it: calls whose work overlaps on the GPU (other streams, other contexts)
 * race.  The context is only read (the call runs its stages on a private
 * view of it that shares the plan), so other calls may use the context
 * meanwhile.  The plan tables are copied into the array from pageable host
 * memory on `stream`, so the call may block the host until those small
 * copies are staged.  A bounded wait that expires inside this call records
 * its code in the context's status word when the context has one, else (a
 * CPDR_FLAG_HOST_ONLY context) in the array's status word, which is cleared
 * at the start of every call: read it with cpdr_check_device_status on the
 * same context and device before the next allocation-free call there.
 */
cpdr_status cpdr_forward_noalloc(const cpdr_ctx *ctx, const void *q, const void *k, const void *v,
                                 const void *beta, const float *gate, void *o, float *final_state, void *stream);

/*
 * Device status: kernels that wait on an mbarrier do so for a bounded number
 * of polls; when a wait gives up, the kernel records a nonzero code in the
 * context's device status word and returns instead of hanging.  This call
 * synchronises `stream`, reads and clears that word, and returns
 * CPDR_ERR_TIMEOUT (with the code in the message) if it was set.  For a
 * context created with CPDR_FLAG_HOST_ONLY, whose kernels can only have run
 * through cpdr_forward_noalloc, it reads and clears the status word of that
 * entry point's array on the current device (CPDR_OK if the entry point has
 * not run on this device).
 */
cpdr_status cpdr_check_device_status(const cpdr_ctx *ctx, void *stream);

/*
 * Self-test of the bounded-wait failure path (no counterpart in the article):
 * launches one warp that waits, for at most `max_cycles` SM clock cycles
 * (0 < max_cycles <= 4e9, about 2 s at the maximum clock), on an mbarrier
 * phase that nothing completes, then records code 1 at site 99 in the
 * context's device status word and returns -- what every bounded wait of the
 * library does when it gives up.  cpdr_check_device_status then reports
 * CPDR_ERR_TIMEOUT and clears the word; the context stays usable.  No fault,
 * trap or unbounded wait is involved.
 */
cpdr_status cpdr_selftest_wait_timeout(const cpdr_ctx *ctx, long long max_cycles, void *stream);

/* Thread-local message for the last non-OK status of this thread. */
const char *cpdr_last_error(void);

/* Library version string. */
const char *cpdr_version(void);

#ifdef __cplusplus
}
#endif
#endif /* CPDR_H_ */
