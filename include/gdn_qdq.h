/*
 * gdn_qdq.h — C ABI of the GB300 (sm_103a) chunked gated delta rule with
 * dynamic fake quantize-dequantize (QDQ) at the recurrent-state and WY "W"
 * sites, and its identity straight-through (STE) backward.
 *
 * Sources of the contract (GatedDeltaNet QAT pull-request pages):
 *   "[1/4] GDN state/W QAT foundation", section "What does this PR do?":
 *       chunk size 64, dynamic FP8 E4M3 fake QDQ at the state and W sites,
 *       identity STE, exact triangular solve, the quantized W saved for
 *       backward; unsupported formats and FP32 inputs are rejected before
 *       launch; BF16 Q/K/V; grouped heads; packed sequences.
 *   same page, section "Usage": state quantizer `axis (0, 1)` with
 *       `state.block_v 64`, W quantizer `axis (0, 1, 2)`.
 *   "[2/4] GDN/KDA decode QAT with INT8 recurrent state", sections "What
 *       does this PR do?" and "Testing": signed symmetric dynamic INT8
 *       (zero point 0, codes in [-127, 127], nearest-even rounding, per-head
 *       [Dk, block_v] scales), gradients through initial states and split
 *       carry, scale arithmetic x * fl(1/s).
 *
 * Conventions that hold for every entry point:
 *   - Every tensor argument is a DEVICE pointer to contiguous row-major
 *     memory owned by the caller.  The library never allocates, frees or
 *     synchronizes; work is enqueued on `stream` (a cudaStream_t passed as
 *     void*, NULL = legacy default stream) and returns before it finishes.
 *   - Arguments are validated on the host before anything is launched; an
 *     invalid call returns a negative gdn_status and enqueues nothing.  No
 *     silent fallback exists: a configuration that is not supported is an
 *     error.  GDN_ERR_CUDA reports a launch failure (cudaGetLastError).
 *   - Notation: B batch rows, T tokens per row, Hk query/key heads, Hv value
 *     heads (Hv % Hk == 0, value head h reads key head h / (Hv / Hk)), Dk key
 *     dim, Dv value dim.  With packed sequences (cu_seqlens != NULL) B == 1,
 *     T is the total token count and N sequences are described by the N+1
 *     int32 offsets of cu_seqlens (device memory, cu[0] == 0, non-decreasing,
 *     cu[N] == T).  Without it N == B and each row is one sequence.
 *   - Chunks are 64 tokens from each sequence's start; a sequence's last
 *     chunk may be shorter.  Per-chunk data is stored at a "chunk slot":
 *       fixed length: slot(n, c) = n * ceil(T / 64) + c,  n_slots = B * ceil(T/64)
 *       packed:       slot(n, c) = floor(cu[n] / 64) + n + c,  n_slots = floor(T/64) + N
 *     (the packed formula is injective for any lengths; unused slots are
 *     left untouched).
 */
#ifndef GDN_QDQ_H_
#define GDN_QDQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GDN_QDQ_ABI_VERSION 7

typedef enum {
  GDN_QDQ_NONE = 0, /* site not quantized                                   */
  GDN_QDQ_E4M3 = 1, /* dynamic FP8 E4M3: s = amax/448, RNE, satfinite      */
  GDN_QDQ_INT8 = 2  /* dynamic signed symmetric INT8: s = amax/127, RNE    */
} gdn_qdq_mode;

typedef enum {
  GDN_DTYPE_BF16 = 0, /* the only accepted q/k/v (and dO) element type    */
  GDN_DTYPE_FP16 = 1, /* rejected                                          */
  GDN_DTYPE_FP32 = 2  /* rejected before launch (first page, "What")       */
} gdn_dtype;

typedef enum {
  GDN_OK = 0,
  GDN_ERR_INVALID_ARG = -1,       /* null pointer, negative size, bad enum   */
  GDN_ERR_UNSUPPORTED_DTYPE = -2, /* q/k/v/dO not bf16                        */
  GDN_ERR_UNSUPPORTED_SHAPE = -3, /* Dk/Dv not 64/128, Hv % Hk, chunk != 64  */
  GDN_ERR_UNSUPPORTED_MODE = -4,  /* QDQ mode or block_v not supported       */
  GDN_ERR_WORKSPACE_TOO_SMALL = -5,
  GDN_ERR_CUDA = -6,              /* a launch failed                         */
  GDN_ERR_MISALIGNED = -7         /* a pointer is not 16-byte aligned        */
} gdn_status;

/* One problem description, shared by the forward and the backward. */
typedef struct {
  int64_t B;                  /* batch rows (1 when packed)                     */
  int64_t T;                  /* tokens per row (total tokens when packed)      */
  int32_t Hk, Hv, Dk, Dv;     /* heads and head dims; Dk, Dv in {64, 128}       */
  int32_t N;                  /* sequences: == B, or packed count (>= 1)        */
  const int32_t* cu_seqlens;  /* device [N + 1] int32, or NULL                  */
  float scale;                /* output scale (1.0 for o_t = S_t q_t)           */
  int32_t state_mode;         /* gdn_qdq_mode at the state site                 */
  int32_t w_mode;             /* gdn_qdq_mode at the W site                     */
  int32_t block_v;            /* state-scale tile width: 16, 32, 64 or 128 (<= Dv) */
  int32_t chunk;              /* chunk length; must be 64                      */
  int32_t dtype;              /* gdn_dtype of q, k, v (and dO); must be BF16    */
  int32_t solve;              /* GDN_SOLVE_EXACT (0): T = (I + A)^-1;
                                 GDN_SOLVE_NEUMANN (1): T = sum_{i<=solve_degree} (-A)^i
                                 ("[7/7] Experimental GDN/KDA approximate-inverse
                                 QAT", "What does this PR do?"), the backward
                                 through that polynomial                       */
  int32_t solve_degree;       /* Neumann degree, 0..63 (63 is already exact)    */
  int32_t save_ctx;           /* 1: the forward writes the context the backward
                                 reads (training); 0: forward only (inference):
                                 `ctx` is scratch for the forward's own launches
                                 and gdn_ctx_bytes() is smaller               */
} gdn_problem;

typedef enum { GDN_SOLVE_EXACT = 0, GDN_SOLVE_NEUMANN = 1 } gdn_solve;

/*
 * Device-side error flag.  Kernels that wait for their own asynchronous
 * copies (TMA transfers signalled on mbarriers) bound every wait; a wait that
 * gives up ends the kernel early and sets this flag, so the outputs of the
 * call that set it are invalid.  Returns the flag (nonzero = a wait gave up)
 * and clears it when `reset` is nonzero; -1 if it cannot be read.  Unlike
 * every other entry point this call synchronizes with the current device.
 */
int gdn_device_error(int reset);

/* Human-readable name of a status code (static string). */
const char* gdn_status_string(int status);

/* GDN_QDQ_ABI_VERSION of the loaded library. */
int gdn_abi_version(void);

/* Host-only validation of a problem description (no CUDA call). */
gdn_status gdn_validate(const gdn_problem* p);

/* Number of chunk slots (see the header comment), or -1 if p is invalid. */
int64_t gdn_num_chunk_slots(const gdn_problem* p);

/*
 * Bytes of the forward's context, or 0 if p is invalid.  With save_ctx = 1
 * it holds what the backward reads (the quantized W and chunk states and the
 * chunk tiles below); with save_ctx = 0 only what the forward's own launches
 * hand to each other.  Segments (each starts on a 256-byte boundary, in this
 * order; gdn_ctx_offset() gives each one's offset, or -1 where absent):
 *   w_codes   u8  [B, T, Hv, Dk]        quantized W codes    (w_mode != NONE)
 *   w_scales  f32 [n_slots, Hv]         W scale per chunk    (w_mode != NONE)
 *   w_full    f32 [B, T, Hv, Dk]        unquantized W        (w_mode == NONE)
 *   cvec      f32 [n_slots, Hv, 5, 64]  per chunk: gamma (in-chunk cumsum of
 *                                       g), e^gamma, e^{gamma_L - gamma}, beta,
 *                                       beta e^gamma (rows past the chunk end:
 *                                       gamma flat, beta 0)
 *   t_img     bf16 [n_slots, Hv, 4096]  T = (I + A)^-1 (lower incl. diagonal)   (save_ctx)
 *   gkk_img   bf16 [n_slots, Hv, 4096]  Gamma o KK^T (strictly lower)           (save_ctx, not fused)
 *   p_img     bf16 [n_slots, Hv, 4096]  P = Gamma o QK^T (lower incl. diagonal) (save_ctx)
 *   d_img     bf16 [n_slots, Hv, Dv/64, 4096]  Delta = U - W^ H^ of each
 *                                       64-column value block        (save_ctx, not fused)
 *             ("fused": Dk = Dv = 128, both sites quantized, block_v 64, exact
 *             solve; that backward recomputes Gamma o KK^T and Delta)
 *             each 64 x 64 tile stored as its shared-memory image: element
 *             (i, j) at i * 64 + 8 * ((j / 8) ^ (i % 8)) + j % 8; rows past
 *             the chunk end are zero (T: identity rows)
 *   tu_img    bf16 [n_slots, Hv, 2, 4096] T diag(beta) split into hi + lo bf16
 *                                       halves (hi = bf16(x), lo = bf16(x - hi)),
 *                                       as images like the tiles above (fused
 *                                       forward only: Dk = Dv = 128, both sites
 *                                       quantized, block_v 64, exact solve)
 *   h_codes   u8  [n_slots, Hv, Dk, Dv] state codes entering each chunk (state_mode != NONE;
 *                                       absent for a forward-only fused call)
 *   h_scales  f32 [n_slots, Hv, Dv/block_v] state scale per [Dk, block_v] tile (as h_codes)
 *   h_full    f32 [n_slots, Hv, Dk, Dv] unquantized state entering each chunk (state_mode == NONE)
 * E4M3 codes are OCP E4M3FN bytes; INT8 codes are two's-complement bytes.
 * Code times scale (fp32 multiply) is the dequantized value; the context
 * therefore holds the quantized W and states exactly.
 */
size_t gdn_ctx_bytes(const gdn_problem* p);

typedef enum {
  GDN_CTX_W_CODES = 0, GDN_CTX_W_SCALES, GDN_CTX_W_FULL, GDN_CTX_CVEC, GDN_CTX_T_IMG,
  GDN_CTX_GKK_IMG, GDN_CTX_P_IMG, GDN_CTX_D_IMG, GDN_CTX_TU_IMG, GDN_CTX_H_CODES,
  GDN_CTX_H_SCALES, GDN_CTX_H_FULL
} gdn_ctx_segment;

/* Byte offset of one context segment (gdn_ctx_segment), or -1 if p is invalid
 * or the segment is absent for this problem. */
int64_t gdn_ctx_offset(const gdn_problem* p, int segment);

/*
 * Forward: o = chunked gated delta rule with state/W fake QDQ.
 *   q, k  bf16 [B, T, Hk, Dk]      v   bf16 [B, T, Hv, Dv]
 *   beta  f32  [B, T, Hv]          g   f32  [B, T, Hv] (log decay, alpha = exp g)
 *   h0    f32  [N, Hv, Dk, Dv] initial state H = S^T, or NULL for zeros
 *   o     f32  [B, T, Hv, Dv]      (written)
 *   ht    f32  [N, Hv, Dk, Dv] final state, unquantized, or NULL (written)
 *   ctx   gdn_ctx_bytes(p) bytes, 256-byte aligned (written; required when
 *         B * T > 0: the forward's launches hand W and the chunk states to
 *         each other through it; with save_ctx = 1 it is also the backward's
 *         context)
 * Per chunk (method of the first page; the pages print no equations, this is
 * the published WY form of the gated delta rule): gamma = in-chunk cumsum of
 * g; A = strictly-lower(beta_i exp(gamma_i - gamma_j) k_i.k_j); T = (I+A)^-1;
 * W = T diag(beta exp(gamma)) K, Q_W over the whole [L, Dk] tile; U = T
 * diag(beta) V; H^ = Q_S(H) per [Dk, 64] tile (h0 included); Delta = U - W^ H^;
 * o = scale (diag(exp(gamma)) Q H^ + (lower-incl(exp(gamma_i-gamma_j) q_i.k_j)) Delta);
 * H <- exp(gamma_L) H^ + (diag(exp(gamma_L - gamma)) K)^T Delta.
 * Three launches: the chunk-local part (A, T, W with its QDQ, U) for all
 * chunks at once, the serial state scan, then the outputs for all chunks at
 * once; `o` holds U after the first launch and Delta (which the scan writes
 * over U) until the last launch writes the outputs over it.
 * A sequence of length 0 returns ht = h0 (not quantized).
 * All pointers must be 16-byte aligned (GDN_ERR_MISALIGNED otherwise).
 * Launches: for Dk = Dv = 128 with both sites quantized, block_v 64 and the
 * exact solve, two: the chunk-local A, T, W (with its QDQ) for all chunks at
 * once, then one fused kernel per (sequence, value head, 64-column value
 * block) that walks the chunks forming U, the state QDQ, Delta, the state
 * update and the outputs on the tensor cores (tcgen05, accumulators in
 * tensor memory).  Otherwise the three launches described above.
 */
gdn_status gdn_chunk_fwd_qdq(const gdn_problem* p, const void* q, const void* k,
                             const void* v, const float* beta, const float* g,
                             const float* h0, float* o, float* ht, void* ctx, void* stream);

/*
 * Scratch bytes the backward needs in its `workspace` argument (caller
 * allocated, 256-byte aligned), or 0 if p is invalid.
 */
size_t gdn_bwd_workspace_bytes(const gdn_problem* p);

/*
 * Backward with identity STE through both QDQ sites (first page, "What":
 * identity straight-through; the quantized W saved by the forward is reused,
 * no second quantizer call).  `ctx` is the forward's context for the same
 * inputs, written with save_ctx = 1 (a problem with save_ctx = 0 is
 * GDN_ERR_INVALID_ARG).  Gradients of L = <dO, o> + <dht, ht>:
 *   dO    bf16 [B, T, Hv, Dv]          dht f32 [N, Hv, Dk, Dv] or NULL (zeros)
 *   dq,dk f32  [B, T, Hk, Dk]  (summed over the value heads sharing a key head)
 *   dv    f32  [B, T, Hv, Dv]          dbeta, dg f32 [B, T, Hv]
 *   dh0   f32  [N, Hv, Dk, Dv] or NULL
 * All outputs are overwritten (not accumulated into).
 */
gdn_status gdn_chunk_bwd_ste(const gdn_problem* p, const void* q, const void* k,
                             const void* v, const float* beta, const float* g, const void* ctx,
                             const void* dO, const float* dht, float* dq, float* dk, float* dv,
                             float* dbeta, float* dg, float* dh0, void* workspace,
                             size_t workspace_bytes, void* stream);

/*
 * Allocation-free backward.  The paper has no counterpart: this is an entry
 * point for callers that cannot allocate device memory when they call the
 * backward (for example a runtime that reserved the device's memory up front
 * for its own pool, or code where an allocation would synchronize the
 * device), so they cannot provide gdn_chunk_bwd_ste's workspace.
 * Same arguments, meaning and results as gdn_chunk_bwd_ste without
 * `workspace` / `workspace_bytes`: the scratch comes from a fixed device array
 * of GDN_NOALLOC_SCRATCH_BYTES inside the library, which every GPU that loads
 * the library holds until the process exits.  Problems whose
 * gdn_bwd_workspace_bytes(p) exceeds that size are rejected before any launch
 * with GDN_ERR_WORKSPACE_TOO_SMALL.  The first call in a CUDA context (on a
 * device, with that device current) looks up the array's device address and
 * keeps it for that context — make it before any stream capture.  Calls share
 * the array, which keeps the last call's contents: every scratch byte a call
 * reads it writes first, so nothing needs clearing; calls that overlap on the
 * GPU race.  Allocates nothing.
 */
#define GDN_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)
gdn_status gdn_chunk_bwd_ste_noalloc(const gdn_problem* p, const void* q, const void* k,
                                     const void* v, const float* beta, const float* g,
                                     const void* ctx, const void* dO, const float* dht, float* dq,
                                     float* dk, float* dv, float* dbeta, float* dg, float* dh0,
                                     void* stream);

/*
 * Standalone fake QDQ of x: a contiguous f32 tensor [batch, rows, cols];
 * one group per (batch index, block of group_cols consecutive columns)
 * spanning all rows — [Dk, 64] state tiles are (rows = Dk, group_cols = 64),
 * a whole-tensor group is (batch = 1, rows = 1, group_cols = cols).
 *   y       f32 like x (written; may alias x)
 *   scales  f32 [batch, cols / group_cols] (written; required)
 *   codes   u8 like x, or NULL (written)
 * Bit-exact definition: a = max|x|; a == 0 gives s = 0, y = x, signed-zero
 * codes; else s = fl(a/M), r = fl(1/s), u = fl(x*r), code = RNE onto the
 * E4M3FN grid with finite saturation (M = 448) or nearest-even integer
 * clamped to [-127, 127] (M = 127), y = fl(code * s).  A nonzero a so small
 * that r overflows (s <= 2^-128, i.e. a up to about M * 2^-128: 1.3e-36 for
 * E4M3, 3.7e-37 for INT8) has no usable scale and is taken like a zero group scaled to zero: s = 0, r = 0,
 * so the codes are signed zeros (INT8: 0) and y = fl(code * 0), a zero of
 * x's sign for E4M3 and +0 for INT8.  The same rule holds at every QDQ site
 * of every entry point.
 */
gdn_status fake_qdq_e4m3(const float* x, float* y, float* scales, uint8_t* codes, int64_t batch,
                         int64_t rows, int64_t cols, int64_t group_cols, void* stream);
gdn_status fake_qdq_int8(const float* x, float* y, float* scales, uint8_t* codes, int64_t batch,
                         int64_t rows, int64_t cols, int64_t group_cols, void* stream);

/*
 * KDA recurrent forward with the state fake QDQ ("[1/4] GDN state/W QAT
 * foundation", "What does this PR do?": KDA has a recurrent reference only;
 * "[2/4] GDN/KDA decode QAT with INT8 recurrent state": the same E4M3 / INT8
 * state quantizer).  The pages print no formula; this is the published Kimi
 * Delta Attention recurrence, i.e. the gated delta rule with one decay per
 * key channel.  Per sequence and value head, with H = S^T (Dk x Dv) starting
 * at h0 and t counted from the sequence start:
 *     if t % p->chunk == 0:  H <- Q(H)   (per [Dk, block_v] tile, as fake_qdq_*)
 *     H <- diag(exp(g_t)) H;  H <- H + beta_t k_t (v_t - H^T k_t)^T;  o_t = scale H^T q_t
 * and ht is the final H, unquantized.
 *   q, k  bf16 [B, T, Hk, Dk]      v  bf16 [B, T, Hv, Dv]     beta f32 [B, T, Hv]
 *   g     f32  [B, T, Hv, Dk]  log decay per key channel
 *   h0    f32  [N, Hv, Dk, Dv] or NULL (zeros)
 *   o     f32  [B, T, Hv, Dv] (written)    ht f32 [N, Hv, Dk, Dv] or NULL (written)
 * The problem description is the chunked forward's, read with these rules:
 * w_mode must be NONE (no W site; GDN_ERR_UNSUPPORTED_MODE), `chunk` is the
 * QDQ period (>= 1; 64 is the chunk-boundary rule, 1 quantizes before every
 * token), block_v is 16, 32 or 64, N <= 65535.  Packed sequences, grouped
 * heads and all alignment rules as for the forward.
 */
gdn_status kda_recurrent_fwd_qdq(const gdn_problem* p, const void* q, const void* k,
                                 const void* v, const float* beta, const float* g,
                                 const float* h0, float* o, float* ht, void* stream);

/*
 * Decode QAT step ("[2/4] GDN/KDA decode QAT with INT8 recurrent state",
 * section "What does this PR do?": after an exact chunked prefill of an
 * explicit prefix, every later token writes the recurrent state through the
 * state quantizer; E4M3 or signed symmetric INT8 with per-head [Dk, block_v]
 * scales; section "Testing": both readouts, split carry, all state scale
 * widths).  The page prints no formula; the step is the chunked forward's
 * chunk-boundary rule with one-token chunks.  Per row b, value head h and
 * token t, with H = S^T (Dk x Dv) and S the carried state:
 *     S^ = Q(S)                 (fake QDQ per [Dk, block_v] tile, exactly as
 *                                fake_qdq_*; skipped when state_mode is NONE)
 *     H  = exp(g) S^ + beta k (v - exp(g) S^^T k)^T
 *     o  = scale H^T q          (readout PRE, as inside a forward chunk)
 *        = scale Q(H)^T q       (readout POST: the state the next token reads)
 *     S <- H                    (carried unquantized)
 * so one call over T tokens equals T one-token calls chained through the
 * state, and the split carry from a prefill is state_in = the forward's ht.
 *   q, k   bf16 [B, T, Hk, Dk]        v bf16 [B, T, Hv, Dv]
 *   beta   f32  [B, T, Hv]            g f32  [B, T, Hv] (log decay)
 *   state_in  f32 [B, Hv, Dk, Dv] carried state, or NULL for zeros
 *   o         f32 [B, T, Hv, Dv] (written)
 *   state_out f32 [B, Hv, Dk, Dv] (written; may BE state_in for an in-place
 *             update, any other overlap is GDN_ERR_INVALID_ARG)
 *   codes     u8  [B, T, Hv, Dk, Dv] codes of S^ read by each token, or NULL
 *   scales    f32 [B, T, Hv, Dv / block_v] scales of S^, or NULL
 * B <= 65535 rows; all pointers 16-byte aligned (GDN_ERR_MISALIGNED).
 * T == 0 copies state_in to state_out.  Host-validated like the forward.
 */
typedef enum { GDN_READOUT_PRE = 0, GDN_READOUT_POST = 1 } gdn_readout;

typedef struct {
  int64_t B;                  /* rows: one sequence and one state each          */
  int64_t T;                  /* tokens per row in this call (>= 0)             */
  int32_t Hk, Hv, Dk, Dv;     /* Dk, Dv in {64, 128}; Hv % Hk == 0              */
  float scale;                /* output scale                                   */
  int32_t state_mode;         /* gdn_qdq_mode of the state                      */
  int32_t block_v;            /* state-scale tile width: 16, 32, 64 or 128, <= Dv */
  int32_t readout;            /* gdn_readout                                    */
  int32_t dtype;              /* gdn_dtype of q, k, v; must be BF16             */
} gdn_decode_problem;

/* Host-only validation of a decode problem (no CUDA call). */
gdn_status gdn_decode_validate(const gdn_decode_problem* p);

gdn_status gdn_decode_qdq(const gdn_decode_problem* p, const void* q, const void* k,
                          const void* v, const float* beta, const float* g,
                          const float* state_in, float* o, float* state_out, uint8_t* codes,
                          float* scales, void* stream);

/*
 * Two-precision GDN forward ("[5/8] ReplaySSM state QAT and two-precision
 * GDN", section "What does this PR do?": an FP32 recurrence anchor and a
 * dynamic FP8 E4M3 read copy grouped by the 128 key channels of each value
 * row; every 16-token flush recomputes the recurrence from the raw inputs and
 * the anchor; read-side quantization errors never overwrite the anchor; GDN
 * with K = 128, FP8 or disabled read quantization).  The page prints no
 * formula; the reading implemented here, per sequence and value head with
 * H = S^T (Dk x Dv), t counted from the sequence start and W = p->flush:
 *     A <- h0 (the anchor), and for each token:
 *     if t % W == 0:  R <- Q_read(A)   (E4M3 fake QDQ, one scale per column of H
 *                                       over all Dk key rows, as fake_qdq_e4m3
 *                                       with rows = Dk, group_cols = 1)
 *     A <- exp(g_t) A;  A <- A + beta_t k_t (v_t - A^T k_t)^T
 *     R <- exp(g_t) R;  R <- R + beta_t k_t (v_t - R^T k_t)^T
 *     o_t = scale R^T q_t
 * and ht = A, the unquantized recurrence.  read_mode NONE makes R = A: the
 * plain gated delta rule token recurrence.
 *   q, k  bf16 [B, T, Hk, 128]     v bf16 [B, T, Hv, Dv]   beta, g f32 [B, T, Hv]
 *   h0    f32  [N, Hv, 128, Dv] or NULL (zeros)
 *   o     f32  [B, T, Hv, Dv] (written)     ht f32 [N, Hv, 128, Dv] or NULL (written)
 *   anchors f32 [gdn_two_precision_anchor_bytes(p) / 4] or NULL: when given, the
 *         anchor A entering every window (the state before token w*W of each
 *         sequence, w = 0, 1, ...) is written there for gdn_two_precision_bwd
 *         (caller allocated; the layout is private to the library)
 * Dk must be 128 (GDN_ERR_UNSUPPORTED_SHAPE), Dv 64 or 128; read_mode NONE or
 * E4M3 (INT8: GDN_ERR_UNSUPPORTED_MODE); flush >= 1; N <= 65535; packed
 * sequences and grouped heads as for the chunked forward; all pointers 16-byte
 * aligned (GDN_ERR_MISALIGNED).
 */
typedef struct {
  int64_t B;                  /* batch rows (1 when packed)                     */
  int64_t T;                  /* tokens per row (total tokens when packed)      */
  int32_t Hk, Hv, Dk, Dv;     /* Dk == 128; Dv in {64, 128}; Hv % Hk == 0       */
  int32_t N;                  /* sequences: == B, or packed count (>= 1)        */
  const int32_t* cu_seqlens;  /* device [N + 1] int32, or NULL                  */
  float scale;                /* output scale                                   */
  int32_t read_mode;          /* gdn_qdq_mode of the read copy: NONE or E4M3    */
  int32_t flush;              /* flush period W in tokens (16 on the page)      */
  int32_t dtype;              /* gdn_dtype of q, k, v; must be BF16             */
} gdn_two_precision_problem;

/* Host-only validation of a two-precision problem (no CUDA call). */
gdn_status gdn_two_precision_validate(const gdn_two_precision_problem* p);

/* Bytes of the forward's anchor buffer: (B*T / W + N) windows' anchors
 * [Hv, 128, Dv] f32, or 0 if p is invalid. */
size_t gdn_two_precision_anchor_bytes(const gdn_two_precision_problem* p);

gdn_status gdn_two_precision_fwd(const gdn_two_precision_problem* p, const void* q,
                                 const void* k, const void* v, const float* beta,
                                 const float* g, const float* h0, float* o, float* ht,
                                 float* anchors, void* stream);

/*
 * Backward of the two-precision profile: the window-wise adjoint (same page
 * and section: "a window-wise adjoint during backward").  Reading implemented:
 * the read copy passes its gradient to the anchor unchanged (identity
 * straight-through estimator at every flush), every other step is
 * differentiated exactly, so for L = <dO, o> + <dht, ht> each window's
 * adjoint runs from its end back to its start through both states, and at the
 * window start the read state's gradient is added to the anchor's.  Each window
 * is recomputed from the anchor the forward saved at its start.
 *   anchors  the forward's (same inputs, same problem, anchors != NULL)
 *   dO    f32 [B, T, Hv, Dv]           dht f32 [N, Hv, 128, Dv] or NULL (zeros)
 *   dq,dk f32 [B, T, Hk, 128]  (summed over the value heads sharing a key head)
 *   dv    f32 [B, T, Hv, Dv]           dbeta, dg f32 [B, T, Hv]
 *   dh0   f32 [N, Hv, 128, Dv] or NULL
 * All outputs are overwritten; the sums over value columns are taken in a fixed
 * order (bitwise repeatable).  Packed sequences must cover tokens 0..T-1.
 * min(flush, T) must be <= 256 (GDN_ERR_UNSUPPORTED_SHAPE), otherwise as the
 * forward.  `workspace`: gdn_two_precision_bwd_workspace_bytes(p) bytes,
 * 256-byte aligned (GDN_ERR_WORKSPACE_TOO_SMALL when smaller).
 */
size_t gdn_two_precision_bwd_workspace_bytes(const gdn_two_precision_problem* p);

gdn_status gdn_two_precision_bwd(const gdn_two_precision_problem* p, const void* q,
                                 const void* k, const void* v, const float* beta,
                                 const float* g, const float* anchors, const float* dO,
                                 const float* dht, float* dq, float* dk, float* dv,
                                 float* dbeta, float* dg, float* dh0, void* workspace,
                                 size_t workspace_bytes, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* GDN_QDQ_H_ */
