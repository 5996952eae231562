/*
 * mtp.h -- C ABI of libmtp: the data-parallel hot path of DeepSeek-V3-style
 * sequential multi-token prediction on NVIDIA GB300 (sm_103a).
 *
 * Sources ("the pages"):
 *   [M7.6] "M7.6 - DeepSeek MTP: Sequential Modules, Teacher Forcing, and
 *          Speculative Runtime" (transformer-system.numinens.com)
 *   [M7.4] "M7.4 - Multi-Token Prediction Foundations" (same site)
 *   [SD]   speculative-decoding page, ailearn.mscapital.top ("投机解码")
 *
 * Conventions shared by every entry point:
 *   - Every tensor pointer is a DEVICE pointer (cudaMalloc / torch CUDA
 *     memory) unless the argument says "host".  Tensors are dense,
 *     row-major, 16-byte aligned.  The caller owns all memory; the library
 *     allocates nothing and keeps no state besides one device error word per
 *     translation unit (read with mtp_check_errors) and the tensor-map
 *     encoder entry point resolved on first use.
 *   - Calls are asynchronous on `stream`.  Inside one call, a GEMM may be
 *     launched as a programmatic dependent of the call's previous kernel (its
 *     setup overlaps that kernel; it reads nothing before it completes); the
 *     first kernel of every call is an ordinary launch, so a call is ordered
 *     after all earlier work on `stream`.  Argument errors are detected on the
 *     host, return a status and launch nothing.  Data-dependent errors (token
 *     id out of range, a kernel wait that ran out of time) set bits of the
 *     device error word (MTP_DEVERR_*) and never trap; spec_verify reports
 *     per-request statuses instead.
 *   - bf16 means IEEE bfloat16 storage with fp32 accumulation.  f32 means
 *     fp32 storage and arithmetic.
 */
#ifndef MTP_H
#define MTP_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MTP_ABI_VERSION 1

typedef enum mtp_status {
  MTP_OK = 0,
  MTP_ERR_INVALID_ARG = 1,  /* null pointer, negative size, bad enum        */
  MTP_ERR_SHAPE = 2,        /* inconsistent dimensions                      */
  MTP_ERR_ALIGNMENT = 3,    /* pointer not 16-byte aligned                  */
  MTP_ERR_WORKSPACE = 4,    /* workspace smaller than the query returned     */
  MTP_ERR_CUDA = 5,         /* a CUDA runtime/driver call failed             */
  MTP_ERR_DEVICE = 6,       /* a kernel set the device error word           */
  MTP_ERR_UNSUPPORTED = 7   /* a shape/dtype combination not implemented  */
} mtp_status;

typedef enum mtp_dtype { MTP_F32 = 0, MTP_BF16 = 1 } mtp_dtype;

/* Denominator policy of each loss term ([M7.6] §0x05).
 * FIXED: every term (main and each depth) divided by B*T, the paper's fixed
 *        denominator for a batch of B packed rows of T positions.
 * MASKED_MEAN: each term divided by its own count of supervised rows; an
 *        empty term is 0 and stays in the D-depth mean ([M7.6] §0x06A). */
/* How the per-depth loss sums S_k (k = 0 main, 1..D depths) and counts N_k
 * become the reported terms L^(k) ("M7.4 - Multi-Token Prediction
 * Foundations" §0x02C names the last four):
 *   FIXED          L^(k) = S_k / n_positions (the paper's 1/T, batch form)
 *   MASKED_MEAN    L^(k) = S_k / N_k          (head mean)
 *   SUM            L^(k) = S_k
 *   GLOBAL         L^(k) = S_k / sum_j N_j    (depths only)
 *   WEIGHTED_PAIR  L^(k) = S_k / sum_j w_j N_j (depths only)
 * and total = L_main + sum_k w_k L^(k), w_k the per-depth weights (lambda/D
 * unless given).  L_main is S_0 / n_positions (FIXED), S_0 (SUM), else
 * S_0 / N_0.  A zero denominator gives 0. */
typedef enum mtp_den {
  MTP_DEN_FIXED = 0,
  MTP_DEN_MASKED_MEAN = 1,
  MTP_DEN_SUM = 2,
  MTP_DEN_GLOBAL = 3,
  MTP_DEN_WEIGHTED_PAIR = 4
} mtp_den;

/* Per-request status written by spec_verify. */
enum {
  MTP_VERIFY_OK = 0,
  MTP_VERIFY_INVALID_DRAFT = 1,   /* draft id outside [0,V) or q_j[y_j] <= 0  */
  MTP_VERIFY_ZERO_RESIDUAL = 2,   /* rejection (or bonus row) with no mass     */
  MTP_VERIFY_INVALID_PROBS = 3,   /* NaN/Inf/negative entry in a row it read   */
  MTP_VERIFY_INVALID_BUDGET = 4,  /* remaining < 1                             */
  MTP_VERIFY_DEVICE_TIMEOUT = 5   /* a bounded wait gave up (also sets the
                                     device error word's MTP_DEVERR_TIMEOUT)  */
};

/* Bits of the device error word. */
enum {
  MTP_DEVERR_TOKEN_RANGE = 1u,  /* a token id outside [0, V) was read (clamped) */
  MTP_DEVERR_TIMEOUT = 2u,      /* a bounded pipeline wait gave up             */
  MTP_DEVERR_SEGMENTS = 4u,     /* a segment id re-appears after another one   */
  /* set beside the condition bits above: which kernel family raised them */
  MTP_DEVERR_FROM_CHAIN = 1u << 8,   /* prologue, norms, segment scan, CE reduce */
  MTP_DEVERR_FROM_GEMM = 1u << 9,    /* tcgen05 GEMM core                        */
  MTP_DEVERR_FROM_ATTN = 1u << 10,   /* chain attention                           */
  MTP_DEVERR_FROM_VERIFY = 1u << 11, /* spec_verify                               */
  MTP_DEVERR_FROM_DRAFT = 1u << 12,  /* draft-step kernels                        */
  MTP_DEVERR_FROM_FP8 = 1u << 13,    /* FP8 block-scaled weight GEMM              */
  MTP_DEVERR_FROM_DGEMM = 1u << 14   /* bf16 decode-shaped GEMM                   */
};

/* Problem sizes of one chain call.
 * B packed rows of T positions; model width d = n_heads * head_dim; SwiGLU
 * width ffn; shared vocabulary V; D sequential MTP depths.  eps is the RMSNorm
 * epsilon (the pages leave it open; 1e-6 recommended).  rope_base > 0 applies
 * rotate-half rotary embedding with that base to q and k at the given
 * positions; 0 disables it.  dtype is an mtp_dtype.
 * bf16 requires d % 128 == 0, head_dim in {64, 128}, ffn % 8 == 0; f32
 * requires head_dim <= 128 and T <= 12800. */
typedef struct mtp_dims {
  int B, T, d, n_heads, head_dim, ffn, V, D;
  float eps;
  float rope_base;
  int dtype;
} mtp_dims;

/* Weights of the chain ([M7.6] §0x03, §0x04B).  Shared by the main head and
 * every depth (passed once): embed [V,d], head [V,d], out_norm [d].
 * Per depth k = 0..D-1, each field below is a HOST array of D device
 * pointers: hnorm, enorm, attn_norm, ffn_norm [d]; eh_proj [d, 2d] whose
 * first d columns multiply the normalised hidden state and last d columns
 * the normalised embedding ("he" order, [M7.6] §0x03, §0x07B); wq, wk, wv,
 * wo [d, d]; w_gate, w_up [ffn, d]; w_down [d, ffn].  Every linear map is
 * y = x W^T (row-major [out, in]).  Element type = dims.dtype. */
typedef struct mtp_weights {
  const void* embed;
  const void* head;
  const void* out_norm;
  const void* const* hnorm;
  const void* const* enorm;
  const void* const* eh_proj;
  const void* const* attn_norm;
  const void* const* wq;
  const void* const* wk;
  const void* const* wv;
  const void* const* wo;
  const void* const* ffn_norm;
  const void* const* w_gate;
  const void* const* w_up;
  const void* const* w_down;
} mtp_weights;

/* Bytes of device workspace mtp_chain_forward / mtp_chain_loss need for
 * these sizes (0 if the sizes are invalid). */
size_t mtp_chain_workspace_bytes(const mtp_dims* dims);

/* Teacher-forced MTP chain, depths 1..D ([M7.6] §0x02-§0x04C, §0x06A).
 * For depth k and position t of packed row b:
 *   h̄ = RMSNorm_{h,k}(h^{k-1}_t), ē = RMSNorm_{e,k}(E[x_{t+k}]),
 *   u = M_k [h̄; ē], a = u + Attn_k(RMSNorm_{a,k}(u)), h^k_t = a + FFN_k(RMSNorm_{f,k}(a))
 * where attention is causal within the segment of t and FFN is SwiGLU.
 * Row t has a state at depth k iff t, ..., t+k are active and in one
 * segment ([M7.6] §0x04C); rows without a state are computed on clamped
 * inputs but their values are undefined.
 *   tokens [B,T] int32 in [0,V) (others set MTP_DEVERR_TOKEN_RANGE and are
 *   clamped); seg [B,T] int32 segment ids, -1 = padding; within a packed row
 *   the ids of successive segments strictly increase (a repeated id sets
 *   MTP_DEVERR_SEGMENTS); pos [B,T] int32 RoPE positions in [0,T), typically
 *   the index within the segment; h0 [B,T,d] main-model hidden states.
 *   h_out [D,B,T,d] receives h^1..h^D (pre-final-norm states).
 *   ws: workspace of at least mtp_chain_workspace_bytes(dims) bytes. */
mtp_status mtp_chain_forward(const mtp_dims* dims, const mtp_weights* w,
                             const int32_t* tokens, const int32_t* seg, const int32_t* pos,
                             const void* h0, void* h_out,
                             void* ws, size_t ws_bytes, cudaStream_t stream);

/* Chain forward plus the shared head and masked cross-entropy
 * ([M7.6] §0x03, §0x05; [M7.4] §0x06F), without materialising logits:
 *   ℓ_t = log Σ_v exp(z_v) - z_label, z = W_U RMSNorm_out(h_t).
 * Term 0 (main) uses h0 with label x_{t+1}, supervised where t+1 is active
 * and in the segment of t; term k uses h^k with label x_{t+k+1}, supervised
 * where t..t+k+1 are active and in one segment.  Then
 *   L = L_main + (lambda / D) Σ_k L^(k), each term reduced by `den`.
 *   sums_counts [2*(D+1)] double: (Σℓ, count) for main, then depths 1..D.
 *   losses [D+2] float: L, L_main, L^(1)..L^(D).
 *   row_loss [(D+1),B,T] float, nullable: ℓ per term and row, NaN where the
 *   row is not supervised.  h_out nullable, as in mtp_chain_forward.
 *   with_main = 0 skips the main term (L_main = 0, its sum/count = 0). */
mtp_status mtp_chain_loss(const mtp_dims* dims, const mtp_weights* w,
                          const int32_t* tokens, const int32_t* seg, const int32_t* pos,
                          const void* h0, float lambda, int den, int with_main,
                          double* sums_counts, float* losses, float* row_loss, void* h_out,
                          void* ws, size_t ws_bytes, cudaStream_t stream);

/* Allocation-free variant of mtp_chain_loss.  The pages have no counterpart:
 * this is an integration entry point.  It is for callers that cannot call
 * cudaMalloc or own device memory for a workspace -- plugin hosts whose
 * allocator belongs to someone else, runtimes that forbid allocation on their
 * hot path, code that must not touch the allocator in the middle of a
 * stream.  Same arguments and results as mtp_chain_loss, without ws/ws_bytes:
 * the workspace is a static device array of MTP_NOALLOC_SCRATCH_BYTES inside
 * the library, held on every GPU that loads the library until the process
 * exits.  Returns MTP_ERR_WORKSPACE, launching nothing, when
 * mtp_chain_workspace_bytes(dims) exceeds that size (small shapes only).  The
 * first call on a device looks up the array's device address with that device
 * current; make that first call before any stream capture.  The address is
 * kept for the life of the process: after cudaDeviceReset of a device, do not
 * call this entry point on that device again.  Calls share the
 * one array: calls that overlap on the GPU race, so serialise them (one
 * stream, or events).  It allocates nothing itself. */
#define MTP_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)
mtp_status mtp_chain_loss_noalloc(const mtp_dims* dims, const mtp_weights* w,
                                  const int32_t* tokens, const int32_t* seg, const int32_t* pos,
                                  const void* h0, float lambda, int den, int with_main,
                                  double* sums_counts, float* losses, float* row_loss, void* h_out,
                                  cudaStream_t stream);

/* Loss assembly from per-term (sum, count) pairs ([M7.6] §0x05, §0x06A):
 * L = L_main + (lambda / D) Σ_k L^(k) with each term reduced by `den`
 * (FIXED divides by n_positions).  A data-parallel caller all-reduces the
 * sums_counts of mtp_chain_loss across ranks first -- numerators and
 * denominators are reduced before dividing -- and passes the global
 * n_positions.  sums_counts [2*(D+1)] double, losses [D+2] float (device). */
mtp_status mtp_loss_assemble(int D, const double* sums_counts, double n_positions, float lambda,
                             int den, int with_main, float* losses, cudaStream_t stream);

/* mtp_loss_assemble with per-depth weights: depth_weights is a HOST array of
 * D floats copied at the call (NULL = lambda/D each; D <= 32 when given). */
mtp_status mtp_loss_assemble_weighted(int D, const double* sums_counts, double n_positions,
                                      const float* depth_weights, float lambda, int den, int with_main,
                                      float* losses, cudaStream_t stream);

/* Exact speculative verification of R requests with gamma drafts each
 * ([M7.6] §0x09 one-proposal selector, generalised to gamma by the
 * left-to-right rule of [SD]).  For j = 0..gamma-1: accept y_j iff
 * u_j < min(1, p_j[y_j] / q_j[y_j]) (evaluated exactly as u_j q_j[y_j] <
 * p_j[y_j]); the first rejection emits a
 * correction drawn from (p_j - q_j)+ / Σ(p_j - q_j)+ and ends the round; an
 * accepted y_j that equals eos, or that fills `remaining`, ends the round
 * with no further token; if all gamma are accepted a bonus is drawn from
 * p_gamma / Σ p_gamma.  A draw from weights w with uniform u' is the smallest
 * index whose running sum exceeds u' Σ w.
 *   p [R, gamma+1, V] f32 target rows; q [R, gamma, V] f32 draft rows;
 *   draft [R, gamma] int32.  Uniforms: Philox4x32-10 with key (seed lo, hi)
 *   and counter (j, r, offset lo, offset hi); word 0 -> accept uniform of
 *   position j, word 1 -> correction/bonus uniform (j = gamma for the bonus);
 *   u = (word >> 8) * 2^-24.
 *   eos [R] nullable (-1 = none); remaining [R] nullable (default gamma+1).
 *   Outputs [R] int32: accepted = number of drafts accepted, next_token =
 *   correction or bonus (-1 if the round ended without one), n_emit =
 *   accepted + (next_token >= 0), status = MTP_VERIFY_*.
 * Reads only p_j[y_j], q_j[y_j] up to the decision and the one row pair (or
 * bonus row) it samples from; those rows are checked for NaN/negatives. */
mtp_status spec_verify(int R, int gamma, int V, const float* p, const float* q,
                       const int32_t* draft, uint64_t seed, uint64_t offset,
                       const int32_t* eos, const int32_t* remaining,
                       int32_t* accepted, int32_t* next_token, int32_t* n_emit,
                       int32_t* status, cudaStream_t stream);

/* Gradient buffers of the training step (fp32, device, same shapes as the
 * corresponding weights; the step ADDS into them, so the caller zeroes them
 * or accumulates across calls).  Per-depth members are host arrays of D
 * device pointers.  NULL members are not computed. */
typedef struct mtp_grads {
  float* embed;     /* [V, d] */
  float* head;      /* [V, d] */
  float* out_norm;  /* [d] */
  float* h0;        /* [B, T, d]: gradient with respect to the main model's hidden states */
  float* const* hnorm;
  float* const* enorm;
  float* const* eh_proj;
  float* const* attn_norm;
  float* const* wq;
  float* const* wk;
  float* const* wv;
  float* const* wo;
  float* const* ffn_norm;
  float* const* w_gate;
  float* const* w_up;
  float* const* w_down;
} mtp_grads;

/* Bytes of device workspace mtp_chain_loss_grad needs (0 if unsupported). */
size_t mtp_chain_grad_workspace_bytes(const mtp_dims* dims);

/* Training step of the chain: mtp_chain_loss's forward (same arguments and
 * outputs, with optional per-depth weights as in mtp_loss_assemble_weighted)
 * followed by the gradients of the assembled loss, added into `grads`
 * ([M7.6] §0x05: the shared head receives the main term's and every depth's
 * gradient).  The head backward recomputes the logits per vocabulary chunk
 * (as [tokens, chunk] for dz = (softmax - onehot) dL/dl and as [chunk,
 * tokens] for dz^T) and never stores them whole.  The module backward then
 * runs depth D down to 1 on activations the forward saved: GEMMs for the
 * weight gradients (on transposed activations) and the input gradients (on
 * transposed weights), SwiGLU from recomputed gate/up pre-activations,
 * segment-causal attention (scores recomputed), RoPE, the norms, and the
 * prologue's two RMSNorms -- the state's into depth k-1, the embedding rows'
 * scattered into grads->embed.  Gradients flow through the bf16 rounding
 * points unchanged.  bf16 only. */
mtp_status mtp_chain_loss_grad(const mtp_dims* dims, const mtp_weights* w, const int32_t* tokens,
                               const int32_t* seg, const int32_t* pos, const void* h0, float lambda, int den,
                               int with_main, const float* depth_weights, double* sums_counts, float* losses,
                               const mtp_grads* grads, void* ws, size_t ws_bytes, cudaStream_t stream);

/* Bytes of device workspace mtp_draft_step needs (0 if the sizes are invalid). */
size_t mtp_draft_workspace_bytes(const mtp_dims* dims);

/* Decode-shaped MTP draft step: one proposal per request ([M7.6] §0x09: a
 * carried-frontier round proposes y from the saved parent hidden state and
 * E(f) and keeps q for verification; §0x09A: the MTP block attends over its
 * own K/V cache).  For request r:
 *   c = [RMSNorm_h(parent_hidden_r); RMSNorm_e(E[frontier_r])], u = M c,
 *   a = u + Attn(RMSNorm_a u) over cached rows [0, ctx_len_r) and the new row
 *   (RoPE at pos_r for its q and k; cached keys are used as stored),
 *   h = a + SwiGLU(RMSNorm_f a), q_r = softmax(W_U RMSNorm_out(h)),
 *   y_r = smallest v with Σ_{i<=v} q_r[i] > u Σ q_r, u = (word 2 >> 8) * 2^-24
 *   of Philox4x32-10 with key (seed lo, hi) and counter (0, r, offset lo, hi).
 * dims: B = R requests (<= 32), T = cache capacity, D = 1, dtype MTP_BF16,
 * d % 64 == 0, head_dim in {64, 128}, ffn % 8 == 0; weights as for the chain
 * (depth arrays of length 1).
 *   parent_hidden [R, d]; frontier [R] int32; pos [R] int32 in [0, T];
 *   kv_k, kv_v [R, T, d] bf16 cached keys/values; ctx_len [R] int32 in [0, T].
 *   q_out [R, V] float receives q; y_out [R] int32 the draws; h_out [R, d]
 *   nullable receives the pre-final-norm state of the new row.
 * Streams the block's weights, the head and the cache once: it is
 * HBM-bandwidth bound. */
mtp_status mtp_draft_step(const mtp_dims* dims, const mtp_weights* w, const void* parent_hidden,
                          const int32_t* frontier, const int32_t* pos, const void* kv_k,
                          const void* kv_v, const int32_t* ctx_len, uint64_t seed, uint64_t offset,
                          float* q_out, int32_t* y_out, void* h_out, void* ws, size_t ws_bytes,
                          cudaStream_t stream);

/* Bytes of device workspace mtp_draft_round needs for `gamma` steps (0 if the
 * sizes are invalid or gamma is outside [1, 31]). */
size_t mtp_draft_round_workspace_bytes(const mtp_dims* dims, int gamma);

/* gamma recurrent draft steps by reuse of one MTP module ([M7.6] §0x09: the
 * retained depth proposes the next token from its own output state).  Step s
 * (0-based) is mtp_draft_step's computation with
 *   parent = h of step s-1 (step 0: parent_hidden), frontier = y of step s-1
 *   (step 0: frontier), position pos_r + s, keys = the cached rows
 *   [0, ctx_len_r), the rows of steps 0..s-1 (their rotated keys and values,
 *   staged in the workspace) and the row itself,
 * and its draw uses word 2 of Philox4x32-10 at counter (s, r, offset lo, hi).
 * The staged rows are not written back to the cache.
 *   q_out [R, gamma, V] float: q of every step (the draft distributions that
 *   spec_verify takes); y_out [R, gamma] int32: the draws (spec_verify's
 *   draft tokens); h_out [R, gamma, d] bf16 nullable: every step's state.
 * gamma in [1, 31]; other arguments as for mtp_draft_step, whose call equals
 * this one with gamma = 1.  The block's weights, the head and the cache are
 * streamed once per step. */
mtp_status mtp_draft_round(const mtp_dims* dims, const mtp_weights* w, const void* parent_hidden,
                           const int32_t* frontier, const int32_t* pos, const void* kv_k, const void* kv_v,
                           const int32_t* ctx_len, int gamma, uint64_t seed, uint64_t offset, float* q_out,
                           int32_t* y_out, void* h_out, void* ws, size_t ws_bytes, cudaStream_t stream);

/* One FP8 block-scaled weight matrix W [n, K] ([M7.6] §0x03C: released
 * weights are FP8 with block scales; the runtime chooses the compute
 * representation).  q: e4m3 codes (OCP FP8 E4M3: sign, 4 exponent bits with
 * bias 7, 3 mantissa bits, subnormals, no infinities, 0x7F/0xFF = NaN),
 * row-major with row stride K bytes, 16-byte aligned; scale: fp32
 * [ceil(n/128), ceil(K/128)] row-major, one factor per 128 x 128 block.
 * The represented weight is W[m][k] = e4m3(q[m][k]) * scale[m/128][k/128],
 * used exactly.  The activations meet it on the tensor cores as e4m3 in two
 * terms: per token and 128-wide k-tile, x~ = 2^E (hi + lo) with 2^E the
 * smallest power of two such that max|x| <= 448 * 2^E, hi = RNE_e4m3(x/2^E),
 * lo = RNE_e4m3(x/2^E - hi); x~ = x for every element of magnitude >=
 * 2^(E-2) and |x~ - x| <= 2^(E-10) otherwise.  Products are summed in fp32,
 * one fp32 partial per 128-wide k-block scaled by its block factors. */
typedef struct mtp_fp8_matrix {
  const void* q;
  const float* scale;
} mtp_fp8_matrix;

/* The linear maps of one MTP module in FP8 (shapes as in mtp_weights:
 * eh_proj [d, 2d], wq/wk/wv/wo [d, d], w_gate/w_up [ffn, d], w_down [d, ffn]). */
typedef struct mtp_block_fp8 {
  mtp_fp8_matrix eh_proj, wq, wk, wv, wo, w_gate, w_up, w_down;
} mtp_block_fp8;

/* mtp_draft_round with the module's linear maps in FP8 block-scaled form
 * ([M7.6] §0x03C; it halves the decode step's weight bytes).
 * w supplies the bf16 embedding, head and norm gains (its linear-map fields
 * are not read and may be null: the output head and norms stay in bf16, as
 * the pages keep them in higher precision); f8 the eight linear maps.
 * Requires ffn % 16 == 0.  Everything else, including the outputs and the
 * random stream, is as for mtp_draft_round. */
mtp_status mtp_draft_round_fp8(const mtp_dims* dims, const mtp_weights* w, const mtp_block_fp8* f8,
                               const void* parent_hidden, const int32_t* frontier, const int32_t* pos,
                               const void* kv_k, const void* kv_v, const int32_t* ctx_len, int gamma,
                               uint64_t seed, uint64_t offset, float* q_out, int32_t* y_out, void* h_out,
                               void* ws, size_t ws_bytes, cudaStream_t stream);

/* Bytes of device workspace mtp_gemm_fp8w needs for reduction length K. */
size_t mtp_gemm_fp8w_workspace_bytes(int K);

/* Diagnostic FP8 weight GEMM (the kernel the FP8 draft step uses):
 * out[R, N] (fp32, row stride N) += x~[R, K] · W^T with W the FP8
 * block-scaled matrix (wq [N, K] e4m3, scale [ceil(N/128), ceil(K/128)]) and
 * x~ the two-term e4m3 form of x (bf16) described at mtp_fp8_matrix.
 * R in [1, 32], K % 16 == 0, x and wq 16-byte aligned; ws: at least
 * mtp_gemm_fp8w_workspace_bytes(K) bytes of device memory, 16-byte aligned. */
mtp_status mtp_gemm_fp8w(int R, int N, int K, const void* x, const void* wq, const float* scale, float* out,
                         void* ws, size_t ws_bytes, cudaStream_t stream);

/* Diagnostic GEMM on the same tcgen05 core the chain uses:
 * C[M,N] (bf16) = A[M,K] (bf16) · B[N,K]^T (bf16), fp32 accumulation.
 * K % 8 == 0; A, B, C 16-byte aligned. */
mtp_status mtp_gemm_bf16(int M, int N, int K, const void* A, const void* B, void* C,
                         cudaStream_t stream);

/* Diagnostic bf16 decode-shaped GEMM (the draft step's linear maps):
 * out[R, N] (fp32, row stride N) += x[R, K] · W^T with x bf16 [R, K] (R in
 * [1, 32]) and W bf16 [N, K]; K % 8 == 0, x and W 16-byte aligned. */
mtp_status mtp_gemm_decode_bf16(int R, int N, int K, const void* x, const void* w, float* out,
                                cudaStream_t stream);

/* Diagnostic fp32-accumulating GEMM on the same core (the training step's
 * gradient GEMMs): out[M,N] (fp32, row stride ldo) += A · B^T, bf16 operands.
 * a_mn = 0: A is row-major [M, K] (row stride lda); a_mn = 1: A is stored as
 * [K, M] (row stride lda), i.e. the product reads the transpose of a
 * row-major [K, M] matrix.  b_mn likewise for B ([N, K] or [K, N]).  K is
 * split into `splits` ranges (1..ceil(K/64)) whose partial tiles are added
 * with fp32 atomics.  Leading dimensions % 8 == 0; pointers 16-byte aligned. */
mtp_status mtp_gemm_f32acc(int M, int N, int K, const void* A, int lda, int a_mn, const void* B, int ldb, int b_mn,
                           float* out, int ldo, int splits, cudaStream_t stream);

/* Failure-path diagnostic of spec_verify's bounded waits (the method has no
 * counterpart; it exercises the failure detection every pipeline wait of
 * this library relies on).  Runs spec_verify's bulk-copy kernel with the same
 * arguments (no EOS, no budget) except that its producer issues no copy, so
 * each request that reaches the row sweep (a rejection or a bonus draw)
 * waits on a ring stage nothing will fill; that wait gives up after
 * `wait_limit_cycles` SM clock cycles (1 .. the library's limit of 3e9,
 * ~1.5 s) with no copy in flight.  Such requests end with status
 * MTP_VERIFY_DEVICE_TIMEOUT, accepted = the accept prefix, next_token = -1,
 * and the device error word gets MTP_DEVERR_TIMEOUT | MTP_DEVERR_FROM_VERIFY
 * (read and cleared by mtp_check_errors); requests that end in the accept
 * phase (invalid draft) report as spec_verify would.  The kernel returns
 * normally and the stream stays usable.  Requires V % 4 == 0 and 16-byte
 * aligned p and q (else MTP_ERR_UNSUPPORTED); other argument errors as
 * spec_verify, plus MTP_ERR_INVALID_ARG for a limit out of range. */
mtp_status mtp_diag_verify_starved(int R, int gamma, int V, const float* p, const float* q,
                                   const int32_t* draft, uint64_t seed, uint64_t offset,
                                   int32_t* accepted, int32_t* next_token, int32_t* n_emit,
                                   int32_t* status, long long wait_limit_cycles, cudaStream_t stream);

/* Kernel classes for mtp_profile_kernel. */
enum {
  MTP_KC_HEAD_CE_GEMM = 0,  /* shared head GEMM with the online max/sum-exp epilogue */
  MTP_KC_GATE_UP_GEMM = 1,  /* gate/up GEMM with the SwiGLU epilogue                 */
  MTP_KC_DOWN_GEMM = 2,     /* down-projection GEMM with the residual epilogue      */
  MTP_KC_QKV_GEMM = 3,      /* QKV GEMM with the RoPE epilogue                      */
  MTP_KC_O_GEMM = 4,        /* attention output GEMM with the residual epilogue     */
  MTP_KC_PROJ_GEMM = 5,     /* eh_proj fusion GEMM                                  */
  MTP_KC_ATTENTION = 6,     /* segment-causal attention                             */
  MTP_KC_SPEC_VERIFY = 7,   /* spec_verify                                          */
  MTP_KC_PROLOGUE = 8,      /* embedding gather + dual RMSNorm + concat of a depth  */
  MTP_KC_COUNT = 9
};

/* Measurement hook (not thread-safe; for benchmarks).  Each kernel class
 * has its own slot.  While a slot is armed, every launch of that class issued
 * by this library records events[2*i] on its stream just before and
 * events[2*i+1] just after the launch, i = 0, 1, ... up to n_pairs;
 * *recorded (host) counts the pairs used.  Events are created by the caller
 * (timing enabled).  A null `events` disarms the slot.  Returns
 * MTP_ERR_INVALID_ARG on a bad class. */
mtp_status mtp_profile_kernel(int kernel_class, cudaEvent_t* events, int n_pairs, int* recorded);

/* Number of kernel launches this library has issued since it was loaded
 * (host-side counter). */
unsigned long long mtp_kernel_launches(void);

/* Synchronises `stream`, ORs the device error words of every kernel file
 * into *flags (host, nullable) and clears them.  Returns MTP_ERR_DEVICE if
 * any bit was set, MTP_ERR_CUDA if the synchronisation failed. */
mtp_status mtp_check_errors(cudaStream_t stream, unsigned int* flags);

/* Static string for a status code. */
const char* mtp_status_string(int status);

/* MTP_ABI_VERSION of the loaded library. */
int mtp_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MTP_H */
