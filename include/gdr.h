/*
 * gdr.h -- C interface of the GB300 (sm_103a) gated delta rule library.
 *
 * The library computes the forward pass of the gated delta rule, the
 * recurrence (state S in R^{d_k x d_v}, one per batch row and head)
 *
 *     S~_t = Diag(alpha_t) S_{t-1},  alpha_t = exp(g_t)
 *     S_t  = S~_t + k_t (z_t - S~_t^T e_t)^T
 *     o_t  = S_t^T (scale * q_t)
 *
 * (Gated DeltaNet-2 notes, key design 1, which names e_t and z_t; state
 * orientation as in LLMs from scratch ch. 11, section 11.1) through the
 * chunkwise WY/UT algorithm with chunks of C = 64 tokens (Gated DeltaNet-2
 * notes, key design 2), plus a single-token recurrent step for decoding.
 * The variant is chosen by flags:
 *
 *   flags                                   e_t                z_t
 *   0                 Gated DeltaNet         beta_t k_t         beta_t v_t
 *   GDR_DECAY_CHANNEL KDA                    beta_t k_t         beta_t v_t
 *   GDR_QMIX          Q-Delta                beta_t (k_t + lam_t q_t)  beta_t v_t
 *   DECAY|ERASE|WRITE Gated DeltaNet-2       b_t (.) k_t        w_t (.) v_t
 *
 * Flags combine independently: the erase input is x_t = k_t + lam_t q_t under
 * GDR_QMIX and k_t otherwise; e_t = b_t (.) x_t under GDR_ERASE_CHANNEL and
 * beta_t x_t otherwise; z_t = w_t (.) v_t under GDR_WRITE_CHANNEL and
 * beta_t v_t otherwise. Gated DeltaNet is the recurrence of LLMs from scratch
 * ch. 11, section 11.2; KDA that of "You could have come up with Kimi Delta
 * Attention", section 4; Q-Delta the rewritten rule of the Q-Delta notes, key
 * design 3.
 *
 * GDR_BETA_CHANNEL selects the README variant of LLMs from scratch ch. 11,
 * section 11.3: the write strength is one value per value channel, beta is
 * [B, T, H, d_v] fp32 (16-byte aligned) and scales the prediction error
 * channel by channel,
 *
 *     S_t = S~_t + k_t (beta_t (.) (v_t - S~_t^T k_t))^T,
 *
 * with one scalar decay per head (g is [B, T, H]). It combines with no other
 * flag (GDR_ERR_UNSUPPORTED) and needs B * H <= 65535. Every column of S then
 * follows its own affine map, so there is no shared (I + T)^{-1}. With bf16
 * inputs and the full workspace (gdr_chunk_fwd_workspace), gdr_chunk_fwd runs
 * it chunkwise on the tensor cores: a preparation kernel writes one packet per
 * chunk (the shared L = tril(decay (.) K K^T, -1), A_qk, the gated q and k, v
 * and beta) into the workspace, and the state pass solves each value column's
 * (I + diag(beta_c) L) W_c = diag(beta_c) R_c by substitution. With fp32
 * inputs or a smaller workspace, gdr_chunk_fwd runs it as a token-order scan
 * with the state in fp32 registers, which needs no workspace;
 * gdr_recurrent_step always takes the token-order form.
 *
 * Conventions common to every call:
 *  - Layouts are dense and row-major. Per-token tensors are [B, T, H, d] with
 *    d fastest; scalar per-token gates are [B, T, H]; states are
 *    [B, H, d_k, d_v] with d_v fastest (S's rows are key channels).
 *  - q, k, v, o, b and w use the call's dtype (fp32 or bf16); g, beta, lam and
 *    the states are always fp32. g is the natural-log decay (alpha = exp(g),
 *    g <= 0 in the pages' usage; any finite value is accepted).
 *  - Ownership: the caller owns and allocates every buffer, workspace
 *    included. The library never allocates or frees device memory and keeps
 *    no per-call state between calls.
 *  - Execution: work is enqueued on `stream` (a cudaStream_t; NULL is the
 *    legacy default stream) and the call returns without synchronising.
 *    Input buffers must stay valid until the work completes.
 *  - Errors: argument errors (null or misaligned pointers, bad sizes or
 *    flags, too small a workspace) are reported synchronously, before
 *    anything is enqueued, and the outputs are left untouched. A launch
 *    failure reported by the CUDA runtime returns GDR_ERR_CUDA. Non-finite
 *    inputs propagate to the outputs; they are not detected.
 *  - Supported sizes: d_k, d_v in {64, 128}; 1 <= B, H <= 65535 (launch grid
 *    extents, GDR_ERR_UNSUPPORTED beyond) and T >= 1 with
 *    B*T*H*max(d_k, d_v) < 2^31 elements per tensor; a ragged last chunk is
 *    handled. 16-byte alignment is required for q, k, v, o, b, w, h0, hT and
 *    state; 4-byte alignment for g, beta and lam.
 *  - Decay range of the chunked path with per-channel gates
 *    (GDR_DECAY_CHANNEL): within one 64-token chunk the summed log-decay of
 *    any key channel must stay above -140 (the chunk algebra factors the decay
 *    of a row pair as e^{G_r - rho} e^{rho - G_i} with rho the half-chunk sum,
 *    and past that the factors leave the fp32 range). The bf16 two-kernel
 *    path checks every chunk: a chunk past the limit makes gdr_chunk_fwd_check
 *    return GDR_ERR_RANGE (detail[0] = b * H + h of the first such sequence
 *    seen, detail[1] = its chunk) and its outputs are not to be used;
 *    gdr_token_fwd computes such inputs without the limit. Scalar
 *    gates, GDR_BETA_CHANNEL and the recurrent step have no such limit.
 *  - Decay range of the chunk backward (every gate variant): within one chunk
 *    the running sum of the log-decay (per key channel, or per row for a
 *    scalar decay) must stay above -80, since the backward's records hold
 *    k / e^{G}. A chunk past it makes gdr_chunk_bwd_check return
 *    GDR_ERR_RANGE (detail as above) and the gradients are not to be used;
 *    gdr_token_bwd computes them without the limit.
 */
#ifndef GDR_H_
#define GDR_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t / CUstream; NULL selects the default stream. */
typedef struct CUstream_st* gdr_stream_t;

typedef enum {
  GDR_OK = 0,
  GDR_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad size or flag */
  GDR_ERR_UNSUPPORTED = 2, /* valid request outside the supported set  */
  GDR_ERR_CUDA = 3,        /* the CUDA runtime reported an error        */
  GDR_ERR_WORKSPACE = 4,   /* workspace missing or smaller than needed  */
  GDR_ERR_TIMEOUT = 5,     /* a bounded device-side wait gave up        */
  GDR_ERR_RANGE = 6        /* channel decay past the chunked range       */
} gdr_status;

typedef enum { GDR_F32 = 0, GDR_BF16 = 1 } gdr_dtype;

enum {
  GDR_DECAY_CHANNEL = 1, /* g is [B,T,H,d_k] (per key channel), else [B,T,H] */
  GDR_ERASE_CHANNEL = 2, /* erase direction b (.) x, b is [B,T,H,d_k]        */
  GDR_WRITE_CHANNEL = 4, /* write vector w (.) v, w is [B,T,H,d_v]           */
  GDR_QMIX = 8,          /* erase input x = k + lam q, lam is [B,T,H]         */
  GDR_BETA_CHANNEL = 16  /* beta is [B,T,H,d_v], scales the error per channel */
};

typedef struct {
  int B, T, H;      /* batch, tokens, heads                                */
  int dk, dv;       /* key and value widths (64 or 128)                    */
  int dtype;        /* gdr_dtype of q, k, v, o, b, w                       */
  unsigned flags;   /* GDR_DECAY_CHANNEL | GDR_ERASE_CHANNEL | ...         */
  float scale;      /* read-out scale on q (d_k^-1/2 in the KDA derivation) */
} gdr_shape;

/* Device workspace bytes for gdr_chunk_fwd on `shape` (may be 0).
 *
 * gdr_chunk_fwd_workspace gives the size that selects the fastest path. For
 * bf16 inputs that is the two-kernel path: one kernel does the intra-chunk
 * work of every chunk of every (batch, head) in parallel and writes a packet
 * per chunk (Q_gamma, -Y, K_tail, A_qk, gamma_C, U: 3 * 128 d_k + 128 d_v +
 * 9216 bytes, 74752 at d_k = d_v = 128) into the workspace; a second kernel
 * runs the state pass over the packets. Total: 256 + B * H * ceil(T / 64) *
 * packet bytes.
 *
 * When B * H is small the state pass, which walks the chunks of each (batch,
 * head) in order, leaves most SMs idle; the full size then also holds the
 * states of a sequence split (see gdr_chunk_fwd_split) and gdr_chunk_fwd uses
 * it when a cost model of the scan passes (waves of 152 CTAs times chunks per
 * run) says it is faster, i.e. when B * H is small against the SM count and
 * the sequences are long; runs hold at least 8 chunks.
 *
 * gdr_chunk_fwd_workspace_min gives the least a call accepts (256 bytes for
 * bf16: the status words). A bf16 call whose workspace is at least that but
 * smaller than the full size runs the single-kernel path, which keeps every
 * intermediate on chip and is slower when B * H is small. Both paths compute
 * the same result up to rounding. fp32 inputs and GDR_BETA_CHANNEL need no
 * workspace.
 *
 * Both return GDR_ERR_INVALID_ARG / GDR_ERR_UNSUPPORTED for a bad shape. */
gdr_status gdr_chunk_fwd_workspace(const gdr_shape* shape, size_t* bytes);
gdr_status gdr_chunk_fwd_workspace_min(const gdr_shape* shape, size_t* bytes);

/*
 * Chunkwise-parallel forward (Gated DeltaNet-2 notes, key design 2; the
 * same WY/UT machinery serves Q-Delta, Q-Delta notes key design 3). For each
 * (batch, head) and each chunk of C = 64 tokens it forms the in-chunk
 * cumulative decay gamma, T = tril(E_bar K_bar^T, -1), A = (I + T)^{-1} by
 * forward substitution, Y = A E_bar and U = A Z, and passes the state across
 * chunks with S_{n+1} = Diag(gamma_C) S_n + K_tail^T (U - Y S_n), reading out
 * O_n = Q_gamma S_n + A_qk (U - Y S_n). The result equals the token
 * recurrence above up to rounding.
 *
 *   q, k   [B,T,H,d_k] dtype      v, o  [B,T,H,d_v] dtype
 *   g      [B,T,H] fp32, or [B,T,H,d_k] under GDR_DECAY_CHANNEL (then
 *          16-byte aligned)
 *   beta   [B,T,H] fp32; required unless both ERASE and WRITE are set
 *          (then ignored); [B,T,H,d_v], 16-byte aligned, under
 *          GDR_BETA_CHANNEL
 *   lam    [B,T,H] fp32; required under GDR_QMIX, ignored otherwise
 *   b      [B,T,H,d_k] dtype; required under GDR_ERASE_CHANNEL, else ignored
 *   w      [B,T,H,d_v] dtype; required under GDR_WRITE_CHANNEL, else ignored
 *   h0     [B,H,d_k,d_v] fp32 initial state, or NULL for the zero state
 *   hT     [B,H,d_k,d_v] fp32 final state (written), or NULL
 *   workspace, ws_bytes: device memory of at least
 *          gdr_chunk_fwd_workspace_min() bytes, 16-byte aligned (NULL allowed
 *          when that is 0); gdr_chunk_fwd_workspace() bytes select the
 *          two-kernel path. It holds the call's status words, which are
 *          cleared on `stream` before the kernels run, and the packets:
 *          calls sharing one workspace must be ordered on the stream.
 *
 * h0 and hT may be the same buffer (streaming: the state read for a (batch,
 * head) is consumed before that (batch, head)'s final state is written); no
 * other output may overlap an input. o is written in dtype, rounded to
 * nearest even for bf16; accumulation and the state are fp32.
 */
gdr_status gdr_chunk_fwd(const gdr_shape* shape, const void* q, const void* k,
                         const void* v, const float* g, const float* beta,
                         const float* lam, const void* b, const void* w,
                         const float* h0, void* o, float* hT, void* workspace,
                         size_t ws_bytes, gdr_stream_t stream);

/*
 * gdr_chunk_fwd with the sequence of every (batch, head) cut into `segments`
 * runs of equal whole chunks (the last may be shorter; fewer runs when there
 * are fewer chunks), bf16 two-kernel path only. The state update is affine in
 * the state, so run p maps its start state by S_end = M_p S_start + H_p, and
 * the maps of consecutive runs compose in order (LLMs from scratch ch. 11,
 * section 11.4). The call runs the chunk preparation once, then one scan pass
 * that gives every run's H_p (from a zero state) and M_p (from the identity,
 * d_k x d_k), a pass that chains the start states S_p = M_{p-1} S_{p-1} +
 * H_{p-1} from h0, and a scan pass of every run from its start state that
 * writes o and, from the last run, hT. The result equals gdr_chunk_fwd up to
 * rounding. segments = 1 is the plain two-kernel path.
 *
 * workspace: at least gdr_chunk_fwd_workspace_split(shape, segments) bytes,
 * else GDR_ERR_WORKSPACE. segments < 1 is GDR_ERR_INVALID_ARG; segments > 1
 * with fp32 or GDR_BETA_CHANNEL, B * segments > 65535, or segments > 1 with
 * B * H > 65535 (launch grid extents) is GDR_ERR_UNSUPPORTED. Other arguments
 * as gdr_chunk_fwd.
 */
gdr_status gdr_chunk_fwd_split(const gdr_shape* shape, int segments, const void* q,
                               const void* k, const void* v, const float* g,
                               const float* beta, const float* lam, const void* b,
                               const void* w, const float* h0, void* o, float* hT,
                               void* workspace, size_t ws_bytes, gdr_stream_t stream);

/* Workspace bytes of gdr_chunk_fwd_split: the two-kernel workspace, then
 * 256-byte aligned per-run buffers (local end states and start states,
 * B * H * segments * d_k * d_v fp32 each; transitions, B * H * segments * d_k *
 * d_k fp32) when segments > 1. */
gdr_status gdr_chunk_fwd_workspace_split(const gdr_shape* shape, int segments,
                                         size_t* bytes);

/*
 * gdr_chunk_fwd for long sequences with few (batch, head) pairs, bf16 only,
 * overlapping the two kernels of the two-kernel path in time. The chunks of
 * every sequence are cut into `segments` time segments of whole chunks (fewer
 * when there are fewer chunks): up to three segments shrink by 5/8 from each to
 * the next, more are equal. The chunk preparation of segment s runs
 * on `stream`; the state pass of segment s runs on `aux_stream` once those
 * packets exist, continuing from the state segment s - 1 left in the
 * workspace, while the preparation of segment s + 1 runs on the SMs the state
 * pass leaves free (it walks the chunks of each (batch, head) in order and
 * takes one SM per (batch, head) at d_k = d_v = 128, per (batch, head, 64
 * value columns) otherwise). The state update and the
 * read-out are those of gdr_chunk_fwd (Gated DeltaNet-2 notes, key design 2);
 * only the order of the launches differs, so the result is the same up to
 * rounding. Each preparation CTA claims one chunk from a counter and exits,
 * so that CTAs come and go and the state pass, which needs a whole SM per CTA,
 * gets its SMs as soon as it may start; give `aux_stream` a higher priority
 * than `stream` (cudaStreamCreateWithPriority) so that its CTAs are scheduled
 * first. `stream` waits for the last state pass before it
 * runs anything enqueued after the call, so results are ordered on `stream`
 * as for gdr_chunk_fwd. `aux_stream` may equal `stream` (no overlap). The call
 * creates and destroys segments + 1 CUDA events (no device memory).
 *
 * workspace: at least gdr_chunk_fwd_workspace_pipelined(shape, segments)
 * bytes, 16-byte aligned (status words, packets, the state between segments,
 * one counter per segment), else GDR_ERR_WORKSPACE; calls sharing one
 * workspace must be ordered. segments outside 1..64 is GDR_ERR_INVALID_ARG;
 * fp32 inputs are GDR_ERR_UNSUPPORTED. Other arguments as gdr_chunk_fwd;
 * gdr_chunk_fwd_check reads its status words.
 */
gdr_status gdr_chunk_fwd_pipelined(const gdr_shape* shape, int segments, const void* q,
                                   const void* k, const void* v, const float* g,
                                   const float* beta, const float* lam, const void* b,
                                   const void* w, const float* h0, void* o, float* hT,
                                   void* workspace, size_t ws_bytes, gdr_stream_t stream,
                                   gdr_stream_t aux_stream);

/* Workspace bytes of gdr_chunk_fwd_pipelined: the two-kernel workspace, then
 * 256-byte aligned the state between segments (B * H * d_k * d_v fp32) and
 * `segments` ints. */
gdr_status gdr_chunk_fwd_workspace_pipelined(const gdr_shape* shape, int segments,
                                             size_t* bytes);

/* The number of time segments gdr_chunk_fwd_pipelined should use on `shape`;
 * 1 means that the overlap is not expected to pay and gdr_chunk_fwd is the
 * call to make. It is above 1 for bf16 when the state pass takes at most half
 * of 152 SMs (its CTAs as above), gdr_chunk_fwd would not split the
 * sequences, and there are at least 64 chunks: up to 8 segments of at least
 * 32 chunks when the state pass takes at most a quarter of the SMs, else up to
 * 3 (one per 32 chunks). */
gdr_status gdr_chunk_fwd_pipeline_segments(const gdr_shape* shape, int* segments);

/*
 * Gradients of the chunked forward (Gated DeltaNet-2 notes, key design 3: the
 * reverse state pass over chunks, the gate-aware dA = dU Z^T + dY E_bar^T and
 * the adjoint of the triangular inverse dT = -tril(A^T dA A^T, -1), then the
 * chain through the decay factors to g, b, w, beta and lam). For the loss
 * L = <dO, o> + <dhT, hT> of gdr_chunk_fwd on the same inputs it writes
 *
 *   dq, dk [B,T,H,d_k] fp32     dv [B,T,H,d_v] fp32
 *   dg     [B,T,H] fp32, or [B,T,H,d_k] under GDR_DECAY_CHANNEL
 *   dbeta  [B,T,H] fp32 (required unless both ERASE and WRITE are set;
 *          [B,T,H,d_v] under GDR_BETA_CHANNEL)
 *   dlam   [B,T,H] fp32 (GDR_QMIX)   db [B,T,H,d_k] fp32 (GDR_ERASE_CHANNEL)
 *   dw     [B,T,H,d_v] fp32 (GDR_WRITE_CHANNEL)
 *   dh0    [B,H,d_k,d_v] fp32, or NULL
 *
 * dO is [B,T,H,d_v] in the call's dtype (16-byte aligned); dhT [B,H,d_k,d_v]
 * fp32 or NULL (zero). Inputs as gdr_chunk_fwd. The arithmetic is fp32 (products
 * on warp-level tensor-core MMAs: split tf32 operands for fp32 inputs, single
 * tf32 products in the per-chunk work for bf16 inputs), through per-chunk
 * records in `workspace` (at least
 * gdr_chunk_bwd_workspace() bytes, 16-byte aligned; about 0.79 MB per chunk at
 * d_k = d_v = 128): the chunk's forward quantities, the state entering and
 * the gradient leaving every chunk. The workspace starts with
 * status words: a chunk whose running log-decay sum falls below -80 (the
 * range of 1 / gamma in fp32) is reported there as GDR_ERR_RANGE, read by
 * gdr_chunk_bwd_check.
 *
 * GDR_BETA_CHANNEL (the write strength per value channel; LLMs from scratch
 * ch. 11, section 11.3) takes a token-order backward instead, the reverse of
 * the recurrence token by token in fp32: the state entering every 64-token
 * chunk is kept on a forward pass, and each chunk is re-run from it before it
 * is walked backward. Its workspace (gdr_chunk_bwd_workspace) holds those
 * states, 64 KB per (batch, head, chunk) at d_k = d_v = 128, and one chunk's
 * states per (batch, head); it has no decay range limit. dq, dk and dg are
 * sums over blocks of 32 value columns, added with atomics, so their last bits
 * may differ between calls; every other output is deterministic.
 */
gdr_status gdr_chunk_bwd_workspace(const gdr_shape* shape, size_t* bytes);
gdr_status gdr_chunk_bwd(const gdr_shape* shape, const void* q, const void* k, const void* v,
                         const float* g, const float* beta, const float* lam, const void* b,
                         const void* w, const float* h0, const void* dO, const float* dhT,
                         float* dq, float* dk, float* dv, float* dg, float* dbeta, float* dlam,
                         float* db, float* dw, float* dh0, void* workspace, size_t ws_bytes,
                         gdr_stream_t stream);

/*
 * Reads the status a gdr_chunk_fwd call left in `workspace` once the work
 * enqueued on `stream` has finished (this call synchronises the stream). It
 * returns GDR_OK; GDR_ERR_TIMEOUT when a bounded device-side wait of that
 * call gave up (the affected outputs are then incomplete; with a non-NULL
 * `detail`, detail[0] receives the index of the CTA that gave up and
 * detail[1] 4 * chunk + the wait); or GDR_ERR_RANGE when a chunk's channel
 * decay was past the limit above (detail as described there). The first
 * report wins. Workspaces of 0 bytes need no check.
 */
gdr_status gdr_chunk_fwd_check(const void* workspace, gdr_stream_t stream,
                               int* detail);

/*
 * gdr_chunk_bwd's gradients walked token by token (the reverse of the
 * recurrence in fp32, no decay factoring): the backward for inputs past the
 * chunk backward's decay range (gdr_chunk_bwd_check returning GDR_ERR_RANGE),
 * the counterpart of gdr_token_fwd. Arguments, outputs and rules as
 * gdr_chunk_bwd; GDR_BETA_CHANNEL takes the same token-order backward as
 * there. A forward pass keeps the state entering every 64-token chunk, and
 * each chunk is re-run from it before it is walked backward; one CTA per
 * (batch, head, 16 value columns), sequential in the tokens, so it is much
 * slower than gdr_chunk_bwd on long sequences. dq, dk, dg, db, dbeta and dlam
 * are sums over the column blocks added with atomics (their last bits may
 * differ between calls); dv, dw and dh0 are deterministic. workspace: at least
 * gdr_token_bwd_workspace() bytes, 16-byte aligned (status words, then the
 * chunk-start states: 64 KB per (batch, head, chunk) at d_k = d_v = 128, and
 * one chunk's states per (batch, head)).
 */
gdr_status gdr_token_bwd_workspace(const gdr_shape* shape, size_t* bytes);
gdr_status gdr_token_bwd(const gdr_shape* shape, const void* q, const void* k, const void* v,
                         const float* g, const float* beta, const float* lam, const void* b,
                         const void* w, const float* h0, const void* dO, const float* dhT,
                         float* dq, float* dk, float* dv, float* dg, float* dbeta, float* dlam,
                         float* db, float* dw, float* dh0, void* workspace, size_t ws_bytes,
                         gdr_stream_t stream);

/*
 * The same for a gdr_chunk_bwd call's workspace: GDR_OK, or GDR_ERR_RANGE
 * when a chunk's log-decay left the backward's range (detail[0] = b * H + h
 * of the first such sequence seen, detail[1] = its chunk). Synchronises
 * `stream`.
 */
gdr_status gdr_chunk_bwd_check(const void* workspace, gdr_stream_t stream,
                               int* detail);

/*
 * gdr_chunk_fwd without a workspace argument, for callers that cannot
 * allocate device memory when they run the forward pass (a plugin whose host
 * framework owns every allocation, a loop where cudaMalloc could block or
 * synchronise the device). It has no counterpart on the pages: it exists for
 * such callers only. The library compiles in a small scratch area (256
 * bytes, the minimum workspace; a shape whose minimum is larger is rejected
 * with GDR_ERR_WORKSPACE) that every GPU using the library holds until the
 * process exits, and passes it where gdr_chunk_fwd takes a workspace, so bf16
 * calls run the single-kernel path; arguments, layouts and results are
 * otherwise those of gdr_chunk_fwd. All calls on a device share that
 * scratch, which keeps what the last call left; each call clears the status
 * words it needs on `stream` first. Calls whose work overlaps on the GPU race
 * on the scratch, so order them on one stream. A device-side timeout is
 * recorded in the scratch; gdr_chunk_fwd_static_check reads it back. The
 * first call on each device looks up the scratch address; make it before any
 * stream capture. `stream` must belong to the current device (else
 * GDR_ERR_INVALID_ARG); a failed lookup or launch clears the cached address,
 * so the first call after cudaDeviceReset looks it up again.
 */
gdr_status gdr_chunk_fwd_static(const gdr_shape* shape, const void* q,
                                const void* k, const void* v, const float* g,
                                const float* beta, const float* lam,
                                const void* b, const void* w, const float* h0,
                                void* o, float* hT, gdr_stream_t stream);

/*
 * The status the last gdr_chunk_fwd_static call on the current device left in
 * the library's scratch, read once the work enqueued on `stream` has finished
 * (this call synchronises the stream), exactly as gdr_chunk_fwd_check reads a
 * workspace: GDR_OK, or GDR_ERR_TIMEOUT with detail[0] the CTA and detail[1]
 * 4 * chunk + the wait. No counterpart on the pages either.
 */
gdr_status gdr_chunk_fwd_static_check(gdr_stream_t stream, int* detail);

/*
 * The same forward (arguments, layouts and results of gdr_chunk_fwd, no
 * workspace) by walking the tokens in order with the fp32 state in registers:
 * S~ = Diag(alpha_t) S, S_t = S~ + k_t (z_t - S~^T e_t)^T, o_t = S_t^T (scale q_t)
 * for each token (LLMs from scratch ch. 11, section 11.2, in the general form
 * of the Gated DeltaNet-2 notes, key design 1). No decay is factored, so any
 * finite log-decay is exact in fp32: this is the path for inputs past the
 * chunked path's channel-decay range (gdr_chunk_fwd_check returning
 * GDR_ERR_RANGE). It is sequential in the tokens, one CTA per (batch, head, 32
 * value columns), and so far slower than the chunked path on long sequences.
 * Every flag; GDR_BETA_CHANNEL takes its own token-order scan. h0 and hT may
 * alias.
 */
gdr_status gdr_token_fwd(const gdr_shape* shape, const void* q, const void* k,
                         const void* v, const float* g, const float* beta,
                         const float* lam, const void* b, const void* w,
                         const float* h0, void* o, float* hT, gdr_stream_t stream);

/*
 * The output epilogue fused into the chunked forward (Gated DeltaNet-2 notes,
 * overall framework, the last stage of its flow chart: the read-out o goes
 * through RMSNorm and the SiLU output gate before the heads merge; LLMs from
 * scratch ch. 11, section 11.3). The result is gdr_rmsnorm_gate applied to the
 * output of gdr_chunk_fwd,
 *
 *   y[b,t,h,c] = o[b,t,h,c] / sqrt(mean_c' o[b,t,h,c']^2 + eps) * weight[c]
 *                * z[b,t,h,c] * sigmoid(z[b,t,h,c]),
 *
 * with o never written: the state pass computes y from its fp32 read-out. It
 * is fused for bf16 inputs with d_k = d_v = 128 and the full workspace (the
 * two-kernel path, whose state pass holds every value column of a row); for
 * every other shape the call runs the forward into y and then the epilogue
 * kernel in place, with the same result up to rounding.
 *
 *   gate->z       [B,T,H,d_v] in the call's dtype, device, 16-byte aligned, apart
 *                 from y
 *   gate->weight  [d_v] fp32 device, 16-byte aligned
 *   gate->eps     finite, >= 0
 *   y             [B,T,H,d_v] in the call's dtype (o's place in gdr_chunk_fwd)
 *
 * Every other argument, the workspace and the errors are those of
 * gdr_chunk_fwd (gdr_chunk_fwd_pipelined for the second form); a null gate or
 * a bad gate argument returns GDR_ERR_INVALID_ARG, d_v other than 64 or 128
 * GDR_ERR_UNSUPPORTED.
 */
typedef struct {
  const void* z;        /* output-gate input, [B,T,H,d_v] */
  const float* weight;  /* RMSNorm gain, [d_v] fp32 */
  float eps;            /* added to the mean square */
} gdr_out_gate;

gdr_status gdr_chunk_fwd_gated(const gdr_shape* shape, const void* q,
                               const void* k, const void* v, const float* g,
                               const float* beta, const float* lam,
                               const void* b, const void* w, const float* h0,
                               const gdr_out_gate* gate, void* y, float* hT,
                               void* workspace, size_t ws_bytes,
                               gdr_stream_t stream);
gdr_status gdr_chunk_fwd_gated_pipelined(const gdr_shape* shape, int segments,
                                         const void* q, const void* k,
                                         const void* v, const float* g,
                                         const float* beta, const float* lam,
                                         const void* b, const void* w,
                                         const float* h0,
                                         const gdr_out_gate* gate, void* y,
                                         float* hT, void* workspace,
                                         size_t ws_bytes, gdr_stream_t stream,
                                         gdr_stream_t aux_stream);

/*
 * One recurrent step for decoding (LLMs from scratch ch. 11, section 11.2,
 * in the general form above; section 11.3 for the streaming protocol: the
 * prefill's final state is the first step's state). shape->T must be 1 and
 * shape->B is the number of sequences N; tensors are the [N,1,H,d] (equally
 * [N,H,d]) slices of the layouts above and the gates likewise (beta is
 * [N,H,d_v] under GDR_BETA_CHANNEL).
 *
 *   state  [N,H,d_k,d_v] fp32, read as S_{t-1} and overwritten with S_t
 *   o      [N,H,d_v] dtype, o_t = S_t^T (scale q_t)
 *
 * Each (sequence, head) reads and writes its state once.
 */
gdr_status gdr_recurrent_step(const gdr_shape* shape, const void* q,
                              const void* k, const void* v, const float* g,
                              const float* beta, const float* lam,
                              const void* b, const void* w, float* state,
                              void* o, gdr_stream_t stream);

/*
 * Chunk-local cumulative log-decay (Gated DeltaNet-2 notes, key design 2:
 * gamma_r = exp(sum_{i<=r} g_i) restarts every chunk; the training-strategy
 * paragraph keeps this sum in fp32). G[b, t, x] = sum of g[b, i, x] over the
 * tokens i <= t of t's chunk (chunks of `chunk` tokens from t = 0), for
 * g, G of shape [B, T, X] fp32 with X = H (scalar gates) or H * d_k
 * (channel gates). chunk must be 64. G may alias g.
 */
gdr_status gdr_gate_cumsum(int B, int T, int X, int chunk, const float* g,
                           float* G, gdr_stream_t stream);

/*
 * Output epilogue after the read-out (Gated DeltaNet-2 notes, overall
 * framework, the last stage of its flow chart; LLMs from scratch ch. 11,
 * section 11.3: RMSNorm, then the SiLU output gate, before the heads merge).
 * For each of `rows` rows of dv channels (rows = B * T * H for o of shape
 * [B,T,H,dv], row-major, no padding):
 *
 *   y[r, c] = o[r, c] / sqrt(mean_c'(o[r, c']^2) + eps) * weight[c]
 *             * z[r, c] * sigmoid(z[r, c])
 *
 *   o, z, y  [rows, dv] in `dtype` (GDR_BF16 or GDR_F32), device, 16-byte
 *            aligned; the arithmetic is fp32 and y is rounded once
 *   weight   [dv] fp32 device, 16-byte aligned: the RMSNorm gain, one value
 *            per value channel, shared by every row
 *   eps      finite, >= 0, added to the mean square (a row of zeros with
 *            eps = 0 yields NaN)
 *
 * y may be o (in place) or z; any other overlap with them returns
 * GDR_ERR_INVALID_ARG, as do null or misaligned pointers (when rows > 0),
 * rows < 0, a bad dtype or a negative or non-finite eps. dv other than 64,
 * 128 or 256 returns GDR_ERR_UNSUPPORTED. rows = 0 launches nothing. The
 * caller owns every buffer; nothing is allocated and the stream is not
 * synchronised.
 */
gdr_status gdr_rmsnorm_gate(long long rows, int dv, gdr_dtype dtype, const void* o,
                            const void* z, const float* weight, float eps, void* y,
                            gdr_stream_t stream);

/* Static, human-readable name of a status code. */
const char* gdr_status_string(gdr_status status);

/* Interface version (incremented on any signature change). */
int gdr_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GDR_H_ */
