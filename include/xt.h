/*
 * xt.h — C ABI of libxt: forward kernels and analytic backward kernels of the ops of a
 * pre-norm transformer block, for one NVIDIA GB300 (sm_103a).
 *
 * Sources (cited by page title and section):
 *   [AE] xtrain "Phase: Autograd Engine + Op Backward — Design Document": op table
 *        (forward / backward of each op), RMSNorm, RoPE, softmax and cross-entropy
 *        derivations, composed attention, tape and gradient accumulation.
 *   [BP] unhomeschool "Träna en språkmodell: Backprop i anpassad CUDA": forward pass of
 *        the GPT-style stack, forward/backward kernel pairs, saved tensors, gradient
 *        buffers with += semantics.
 *   [DO] xtrain "Phase T18: Dropout (device RNG + mask) — Design Document": counter-based
 *        RNG, per-site seeds, train/eval switch, residual-path wiring.
 *
 * Conventions shared by every entry point
 *   - Return value: XT_OK (0) or an xt_status code; xt_last_error() gives a message
 *     (thread-local, valid until the next call on the same thread).
 *   - Pointers: DEVICE pointers owned by the caller, unless a comment says "host".
 *     The library never allocates or frees memory.  Scratch space ("ws") is caller
 *     memory of at least the size the matching *_workspace_size() reports; its contents
 *     on entry do not matter, except for the matmul and block workspaces, whose first
 *     4096 bytes must be zero before their first use (every call leaves them zero).
 *   - stream: a cudaStream_t passed as void* (NULL = legacy default stream).  Every call
 *     only enqueues work on it and returns; nothing synchronises, except
 *     xt_get_device_errors().
 *   - Layout: row-major, contiguous unless a leading dimension (ld, in elements) is given.
 *     "rows, cols": x is [rows, cols].  Weights are [in, out] and a linear layer is y = x @ W.
 *   - dtype: XT_F32 or XT_BF16 storage; arithmetic is float32 (GEMMs: tf32 or bf16
 *     tensor-core products with float32 accumulation).  Saved statistics (inv_rms, mean,
 *     rstd, lse) are always float32.  Token ids and targets are int32.
 *   - accumulate flags: 0 ⇒ dst = g; 1 ⇒ dst += g ([AE] § 梯度累加: first push sets,
 *     later pushes add; [BP] § Ackumulation över mikrobatcher: backward adds into the
 *     gradient buffers).
 *   - Vector paths need 16-byte aligned pointers; misaligned pointers are still handled
 *     (a scalar path) unless a function says otherwise.  Sizes are validated on the host;
 *     invalid arguments return XT_ERR_INVALID_ARG before anything is launched.
 *   - Errors detected on the device (an id or target outside [0, V), a bounded wait that
 *     gave up) set bits in a device flag word read by xt_get_device_errors(); the offending
 *     element is skipped (its output row is written as NaN where one exists).
 */
#ifndef XT_H
#define XT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  XT_OK = 0,
  XT_ERR_INVALID_ARG = 1,
  XT_ERR_UNSUPPORTED = 2,
  XT_ERR_ALIGNMENT = 3,
  XT_ERR_CUDA = 4,
  XT_ERR_TIMEOUT = 5
} xt_status;

typedef enum { XT_F32 = 0, XT_BF16 = 1 } xt_dtype;

/* device error flag bits */
#define XT_DEVERR_INDEX 1u   /* a token id or target outside [0, V) */
#define XT_DEVERR_TIMEOUT 2u /* a bounded mbarrier wait in a GEMM gave up */

const char* xt_last_error(void);
const char* xt_version(void);

/* Synchronises `stream`, then copies the device flag word to *out (host pointer).
 * Returns XT_ERR_TIMEOUT if the timeout bit is set, XT_OK otherwise. */
int xt_get_device_errors(uint32_t* out, void* stream);
int xt_clear_device_errors(void* stream);

/* Number of CUDA kernels libxt has launched in this process (host-side counter). */
uint64_t xt_launch_count(void);

/* Limit, in nanoseconds, of the bounded waits inside the tensor-core kernels (the GEMM and the
 * fused attention) on work from their other roles: TMA copies landing, MMAs completing, an
 * accumulator being drained, a stream-K partial being published.  A wait that runs out sets
 * XT_DEVERR_TIMEOUT in the device flag; the kernel then stops issuing work, waits (with the
 * default limit) for the copies and MMAs it already issued, releases its tensor memory and
 * returns, so the context stays usable.  Process-wide; read when a launch is enqueued (a
 * captured graph keeps the value it was captured with).  ns = 0 restores the default of 2 s.
 * Limits under 1 ms poll without suspending (for tests of the give-up paths).  After a
 * give-up the outputs are undefined, and a stream-K matmul workspace may hold stale flag
 * words: zero it before its next use.  Always returns XT_OK. */
int xt_set_wait_limit_ns(uint64_t ns);
uint64_t xt_get_wait_limit_ns(void);

/* GEMM timing for measurement: with capacity > 0, the next `capacity` GEMM launches each get
 * a record tagged with its algorithmic FLOPs (2·M·N·K per batch; for the causal modes only the
 * unmasked half) and a region of a device buffer in which every CTA of the GEMM kernel (and of
 * a K split's reduce kernel) writes %globaltimer when it starts work (after its wait for the
 * preceding kernel) and when it has finished.  No event or extra node enters the stream, so the
 * launches keep their programmatic dependent-launch overlap.  The buffer (capacity × 32 KB) is
 * allocated by this call on the current device, not during the launches; capacity 0 disables
 * recording (the buffer is kept for reuse).  Launches captured into a CUDA graph keep their
 * region, so every replay rewrites it (the read returns the latest replay's timings); a graph
 * captured with profiling on should not be replayed after a later xt_profile_gemm call.
 * xt_profile_gemm_read
 * synchronises the device and copies up to max_records records into host arrays: flops,
 * milliseconds (latest end minus earliest start over the record's CTAs), and (if shapes !=
 * NULL) 8 ints per record: M, N, K, batches, tile width BN (1000 + BN for the paired-CTA
 * kernel), A MN-major, B MN-major, schedule code (causal mode, 10 × K splits, 1000 for
 * stream-K over every unit, 1000 + s for s lockstep K slices).  *n receives the number
 * recorded. */
int xt_profile_gemm(int capacity);
int xt_profile_gemm_read(double* flops, float* ms, int* shapes, int max_records, int* n);

/* ---------------------------------------------------------------------------------
 * Gradient accumulation ([AE] § 梯度累加, push_grad/accumulate): dst[i] += src[i].
 * dst and src may have different dtypes (e.g. bf16 src into an f32 dst).
 * ------------------------------------------------------------------------------- */
int xt_accumulate(void* dst, int dt_dst, const void* src, int dt_src, int64_t n, void* stream);
/* dst[i] = src[i] converted between dtypes (bf16 results round to nearest even). */
int xt_convert(void* dst, int dt_dst, const void* src, int dt_src, int64_t n, void* stream);

/* ---------------------------------------------------------------------------------
 * Elementwise ops, [AE] op table rows add / mul / scale.  n elements, one dtype.
 * Backward grads may be NULL to skip them.
 * ------------------------------------------------------------------------------- */
int xt_add_fwd(const void* a, const void* b, void* y, int64_t n, int dt, void* stream);
/* da = d, db = d (copy or accumulate) */
int xt_add_bwd(const void* d, void* da, void* db, int64_t n, int dt, int acc_a, int acc_b,
               void* stream);
int xt_mul_fwd(const void* a, const void* b, void* y, int64_t n, int dt, void* stream);
/* da = d∘b, db = d∘a.  a and b may be the same pointer (mul(x, x)). */
int xt_mul_bwd(const void* d, const void* a, const void* b, void* da, void* db, int64_t n,
               int dt, int acc_a, int acc_b, void* stream);
int xt_scale_fwd(const void* x, void* y, int64_t n, float alpha, int dt, void* stream);
/* dx = d·alpha */
int xt_scale_bwd(const void* d, void* dx, int64_t n, float alpha, int dt, int acc, void* stream);

/* Full sum to one float32 (device pointer `out`), deterministic two-stage reduction.
 * Needed by the validation loss L = Σ W∘out ([AE] § 验证方法). */
int xt_sum_workspace_size(int64_t n, size_t* bytes);
int xt_sum_fwd(const void* x, int64_t n, int dt, float* out, void* ws, void* stream);
/* dx[i] = *upstream (device float32 scalar) */
int xt_sum_bwd(const float* upstream, void* dx, int64_t n, int dt, int acc, void* stream);

/* ---------------------------------------------------------------------------------
 * add_bias ([AE] op table row add_bias): y[r,c] = x[r,c] + bias[c];
 * backward dx = d (if dx != NULL), dbias[c] = Σ_r d[r,c], summed in a fixed order
 * (per-CTA partials in ws, then one ordered pass).  bias / dbias have dtype dt_bias.
 * ------------------------------------------------------------------------------- */
int xt_colsum_workspace_size(int64_t rows, int64_t cols, size_t* bytes);
int xt_add_bias_fwd(const void* x, const void* bias, void* y, int64_t rows, int64_t cols, int dt,
                    void* stream);
int xt_add_bias_bwd(const void* d, void* dx, void* dbias, int64_t rows, int64_t cols, int dt,
                    int dt_bias, void* ws, int acc_dx, int acc_dbias, void* stream);

/* ---------------------------------------------------------------------------------
 * Activations.  silu ([AE] op table row silu): y = x·σ(x), dx = d·(σ + x·σ·(1−σ)).
 * swiglu ([AE] op table row swiglu): y = silu(g)∘u with g the gate; g and u may be
 * column blocks of one buffer (row strides ld_in), grads likewise (ld_grad).
 * gelu (exact, erf form; [BP] § kernel-pair table, k_mlp_fwd/bwd; backward reads the saved
 * pre-activation, [BP] § Sparade tensorer): y = x·Φ(x), dx = d·(Φ(x) + x·φ(x)).
 * ------------------------------------------------------------------------------- */
int xt_silu_fwd(const void* x, void* y, int64_t n, int dt, void* stream);
int xt_silu_bwd(const void* d, const void* x, void* dx, int64_t n, int dt, int acc, void* stream);
int xt_swiglu_fwd(const void* g, const void* u, int64_t ld_in, void* y, int64_t ld_out,
                  int64_t rows, int64_t cols, int dt, void* stream);
int xt_swiglu_bwd(const void* d, int64_t ld_d, const void* g, const void* u, int64_t ld_in,
                  void* dg, void* du, int64_t ld_grad, int64_t rows, int64_t cols, int dt,
                  int acc, void* stream);
int xt_gelu_fwd(const void* x, void* y, int64_t n, int dt, void* stream);
int xt_gelu_bwd(const void* d, const void* x, void* dx, int64_t n, int dt, int acc, void* stream);

/* ---------------------------------------------------------------------------------
 * RMSNorm ([AE] § RMSNorm): ir = 1/√(mean_c x² + eps), y = x·ir·γ, inv_rms[r] = ir saved.
 * Backward, g = d∘γ: dx = ir·g − x·ir³/n·Σ_c g·x; dγ[c] = Σ_r d·x·ir.
 * d, x, gamma have dtype dt; dx has dtype dt_dx (dt, or XT_F32 with bf16 inputs: a float32
 * residual-gradient buffer); dgamma has dtype dt_param.  dx or dgamma may be NULL.
 * ------------------------------------------------------------------------------- */
int xt_norm_bwd_workspace_size(int64_t rows, int64_t cols, size_t* bytes);
int xt_rms_norm_fwd(const void* x, const void* gamma, void* y, float* inv_rms, int64_t rows,
                    int64_t cols, float eps, int dt, void* stream);
int xt_rms_norm_bwd(const void* d, const void* x, const void* gamma, const float* inv_rms,
                    void* dx, void* dgamma, int64_t rows, int64_t cols, int dt, int dt_dx,
                    int dt_param, void* ws, int acc_dx, int acc_param, void* stream);

/* Allocation-free variant of xt_rms_norm_bwd (the pages have no counterpart: it exists for
 * callers, not for the method).  Some callers cannot allocate device memory where they run
 * the backward: for example a plug-in inside a host framework that owns all device memory
 * through its own pool and hands out no scratch, or a latency-critical loop in which
 * cudaMalloc (which can synchronise the device) is not allowed.  They still pass d, x, gamma,
 * inv_rms, dx and dgamma as for xt_rms_norm_bwd; the dγ partial sums go to a fixed scratch
 * array inside libxt instead of a ws buffer.  Results equal xt_rms_norm_bwd's up to the
 * summation order of dγ (at most 128 partial rows here).
 *   - Limit: cols ≤ 8192 (else XT_ERR_UNSUPPORTED); the scratch is 128 × 8192 floats (4 MiB),
 *     held by every GPU that loads libxt until the process exits.
 *   - The first call on each device looks the scratch's device address up with that device
 *     current (cudaGetSymbolAddress); make that first call before any stream capture.  The
 *     address is kept for the life of the process: after cudaDeviceReset on a device (which
 *     reloads libxt's device code there, possibly elsewhere) do not call this entry point on
 *     that device again in the same process.
 *   - At most 128 blocks walk the rows (the scratch holds one partial row per block), against
 *     up to 4 per SM for xt_rms_norm_bwd: on long inputs it is correspondingly slower.
 *   - No cudaMalloc, cudaFree or allocating library routine is called.  Nothing in the
 *     scratch needs to start at zero: each call overwrites every partial row it reads.
 *   - All calls share the one array: calls that overlap on the GPU (several streams or host
 *     threads) race on it and must be serialised by the caller. */
int xt_rms_norm_bwd_noalloc(const void* d, const void* x, const void* gamma, const float* inv_rms,
                            void* dx, void* dgamma, int64_t rows, int64_t cols, int dt, int dt_dx,
                            int dt_param, int acc_dx, int acc_param, void* stream);

/* LayerNorm (standard definition; [BP] § kernel-pair table k_layernorm_fwd/bwd and
 * § Sparade tensorer: mean and variance saved — saved here as mean and rstd):
 * μ = mean x, var = mean (x−μ)², rstd = 1/√(var+eps), x̂ = (x−μ)·rstd, y = x̂·γ + β.
 * Backward, g = d∘γ: dx = rstd·(g − mean g − x̂·mean(g∘x̂)); dγ = Σ_r d∘x̂; dβ = Σ_r d.
 * Dtypes as for xt_rms_norm_bwd. */
int xt_layernorm_fwd(const void* x, const void* gamma, const void* beta, void* y, float* mean,
                     float* rstd, int64_t rows, int64_t cols, float eps, int dt, void* stream);
int xt_layernorm_bwd(const void* d, const void* x, const void* gamma, const float* mean,
                     const float* rstd, void* dx, void* dgamma, void* dbeta, int64_t rows,
                     int64_t cols, int dt, int dt_dx, int dt_param, void* ws, int acc_dx,
                     int acc_param, void* stream);

/* ---------------------------------------------------------------------------------
 * RoPE ([AE] op table row rope and § RoPE 反向推导): for each pair (i, i+h), h = hd/2,
 * θ = s·base^(−2i/hd):  y_i = x_i cos θ − x_{i+h} sin θ;  y_{i+h} = x_{i+h} cos θ + x_i sin θ.
 * Backward is the transposed rotation: dx_i = d_i cos + d_{i+h} sin, dx_{i+h} = d_{i+h} cos − d_i sin.
 * xt_rope_table fills table[2][S][hd/2] (cos then sin, float32, angles in float64) for
 * positions pos_offset + s.  Token (b, s) head h lives at x + (b·S + s)·ld + h·hd.
 * x and y may alias (in place).  hd must be even.
 * ------------------------------------------------------------------------------- */
int xt_rope_table(float* table, int S, int hd, double base, int pos_offset, void* stream);
int xt_rope_fwd(const void* x, void* y, const float* table, int B, int S, int H, int hd,
                int64_t ld, int dt, void* stream);
int xt_rope_bwd(const void* d, void* dx, const float* table, int B, int S, int H, int hd,
                int64_t ld, int dt, int acc, void* stream);

/* ---------------------------------------------------------------------------------
 * Row-wise safe softmax ([AE] op table row softmax and § Softmax 反向推导):
 * y = exp(x − max)/Σ exp(x − max); dx = y∘(d − Σ_c d∘y).
 * causal: 0 = no mask; 1 = row r is query s = r mod q_len and columns c > s are masked
 * (y = 0 there, written); 2 = as 1, but only columns c < min(cols, 128·(⌊s/128⌋+1)) are
 * read or written (the layout the causal attention GEMMs consume; entries beyond are
 * left untouched).
 * ------------------------------------------------------------------------------- */
int xt_softmax_fwd(const void* x, void* y, int64_t rows, int64_t cols, int causal, int64_t q_len,
                   int dt, void* stream);
int xt_softmax_bwd(const void* d, const void* y, void* dx, int64_t rows, int64_t cols, int causal,
                   int64_t q_len, int dt, int acc, void* stream);

/* ---------------------------------------------------------------------------------
 * Fused attention ([AE] § Attention 用组合: per (batch, head) scores = Q Kᵀ·(1/√hd),
 * P = softmax(scores), O = P V; backward dV = Pᵀ dO, dP = dO Vᵀ, dS = softmax_bwd(dP, P),
 * dQ = dS K·(1/√hd), dK = dSᵀ Q·(1/√hd)), computed tile by tile on the tensor cores without
 * writing P: the same values as the composition up to rounding (P is rounded to bf16 before
 * it multiplies V, as in the composed bf16 path).
 *
 * Layout: token t = b·S + s is row t of each matrix; head h of q, k, v occupies columns
 * [h·hd, h·hd + hd) of its row, rows ld_qkv elements apart (q, k, v may be column blocks of
 * one [T, 3·H·hd] buffer); o and d_o likewise with ld_o; dq, dk, dv with ld_dqkv.
 * causal: 1 masks key c from query s when c > s (the masked probabilities are 0); 0 none.
 * lse (float32 [B][H][S], written by the forward, read by the backward) is the natural-log
 * normaliser log Σ_c exp(scores[s, c]) over the visible keys.
 * dq, dk, dv are overwritten.  The backward's workspace (xt_attention_bwd_workspace_size)
 * holds D = Σ_c dO∘O per (b, h, s).  o_lo (optional, may be NULL; bf16, the layout and row
 * stride of o) receives O − bf16(O) rounded to bf16, so o + o_lo holds O to ~2⁻¹⁶ relative;
 * passed to the backward it is part of the O that D is formed from, which keeps the rows of
 * dS summing to ~0 (with the bf16 O alone they carry its 2⁻⁹ rounding as a bias).
 * Supported: dt = XT_BF16, hd = 64, row strides multiples of 8 elements, all pointers
 * 16-byte aligned (else XT_ERR_UNSUPPORTED / XT_ERR_ALIGNMENT).  Device-side waits are
 * bounded; on expiry XT_DEVERR_TIMEOUT is set in the device error flag.
 * ------------------------------------------------------------------------------- */
int xt_attention_fwd(const void* q, const void* k, const void* v, int64_t ld_qkv, void* o, void* o_lo,
                     int64_t ld_o, float* lse, int B, int S, int H, int hd, int causal, int dt, void* stream);
int xt_attention_bwd_workspace_size(int B, int S, int H, size_t* bytes);
int xt_attention_bwd(const void* q, const void* k, const void* v, int64_t ld_qkv, const void* o,
                     const void* o_lo, const void* d_o, int64_t ld_o, const float* lse, void* dq, void* dk,
                     void* dv, int64_t ld_dqkv, void* ws, size_t ws_bytes, int B, int S, int H, int hd,
                     int causal, int dt, void* stream);

/* ---------------------------------------------------------------------------------
 * Cross-entropy, mean over rows ([AE] op table row cross_entropy, § Cross-entropy 反向推导):
 * loss = (1/R) Σ_r (lse_r − x[r, t_r]);  dx = upstream·(softmax(x_r) − onehot(t_r))/R.
 * lse (float32 [rows]) is saved by the forward; `loss` and `upstream` are device float32
 * scalars.  dlogits may alias logits (in place) when dt_grad == dt.
 * ------------------------------------------------------------------------------- */
int xt_cross_entropy_workspace_size(int64_t rows, size_t* bytes);
/* Forward and backward in one pass over the logits (for the loss at the root of a training
 * graph): the results of xt_cross_entropy_fwd followed by xt_cross_entropy_bwd with acc = 0
 * (lse, loss, dlogits; dlogits may be logits), up to float32 summation order.  Each row is
 * held in shared memory while its lse and gradient are formed, so the logits are read from
 * HBM once.  Rows of more than 200 KB (e.g. 128256 bf16 logits) are split across a cluster of
 * 2, 4 or 8 CTAs, each holding its chunk of the row; the chunks' (max, Σ exp) pairs are
 * exchanged through distributed shared memory and merged in rank order.  Rows whose length
 * is not a multiple of 16 bytes, or buffers not 16-byte aligned, take the two-kernel path. */
int xt_cross_entropy_fwd_bwd(const void* logits, const int32_t* targets, float* lse, float* loss,
                             const float* upstream, void* dlogits, int64_t rows, int64_t V, int dt,
                             int dt_grad, void* ws, void* stream);
int xt_cross_entropy_fwd(const void* logits, const int32_t* targets, float* lse, float* loss,
                         int64_t rows, int64_t V, int dt, void* ws, void* stream);
/* The fan-out of [AE] § 梯度累加 fused: one logits tensor x [rows, V] consumed by three ops
 * whose scalar results are added, L = CE(x) + c_lin·Σx + c_sq·Σ(x∘x), forward and backward in
 * one pass over x.  The gradient is the sum of the three consumers' contributions times the
 * upstream gradient u of L (device float32 scalar; NULL means 1, the loss at the root):
 *   grad (+)= u·((softmax(x_r) − onehot(t_r))/rows + c_lin + 2·c_sq·x)   (float32, [rows, V]),
 * written once (acc = 1 adds it to grad's contents: later pushes add).  Outputs (device
 * float32): loss = CE mean, sums[0] = Σx, sums[1] = Σx², sums[2] = L; lse [rows].  Rows are
 * split across a cluster of CTAs as in xt_cross_entropy_fwd_bwd; V·element size must be a
 * multiple of 16 bytes and logits / grad 16-byte aligned (XT_ERR_ALIGNMENT).  ws:
 * xt_cross_entropy_fanout_workspace_size bytes.  A target outside [0, V) sets XT_DEVERR_INDEX
 * and makes that row's loss term and gradient NaN. */
int xt_cross_entropy_fanout_workspace_size(int64_t rows, size_t* bytes);
/* Process-wide override of how the one-pass cross-entropy splits wide rows: clusters of cl ∈
 * {1, 2, 4, 8} CTAs with nb ∈ {1, 2} chunk buffers each (where the chunks fit), or (0, 0) for
 * the automatic choice (default).  For measurement and tests; XT_ERR_INVALID_ARG otherwise. */
int xt_ce_set_split(int cl, int nb);
int xt_cross_entropy_fanout_fwd_bwd(const void* logits, const int32_t* targets, float c_lin, float c_sq,
                                    const float* upstream, float* lse, float* loss, float* sums, void* grad,
                                    int acc, int64_t rows, int64_t V, int dt, void* ws, size_t ws_bytes,
                                    void* stream);
int xt_cross_entropy_bwd(const void* logits, const int32_t* targets, const float* lse,
                         const float* upstream, void* dlogits, int64_t rows, int64_t V, int dt,
                         int dt_grad, int acc, void* stream);

/* ---------------------------------------------------------------------------------
 * Inverted dropout with a counter-based mask ([DO] § RNG：counter-based, § dropout 节点的
 * backward): for flat element index i (uint64),
 *   key = seed ⊕ (i·0x9E3779B97F4A7C15), h = splitmix64(key), u = (h>>40)·2⁻²⁴ (float32),
 *   keep = u ≥ p, y = keep ? x·scale : 0 with scale = float32(1/(1−p)).
 * The backward regenerates the same mask from (seed, i).  p == 0 or training == 0 is an
 * exact copy.  p must be in [0, 1).  xt_dropout_mask writes the keep mask (1/0 bytes).
 * xt_dropout_add_fwd fuses the residual: out = h + dropout(a) (out may alias h).
 * ------------------------------------------------------------------------------- */
int xt_dropout_fwd(const void* x, void* y, int64_t n, float p, uint64_t seed, int training,
                   int dt, void* stream);
int xt_dropout_bwd(const void* d, void* dx, int64_t n, float p, uint64_t seed, int training,
                   int dt, int acc, void* stream);
/* Same, with d of dtype dt_d (e.g. a float32 residual gradient) and dx of dtype dt_dx. */
int xt_dropout_bwd_ex(const void* d, int dt_d, void* dx, int dt_dx, int64_t n, float p,
                      uint64_t seed, int training, int acc, void* stream);
int xt_dropout_mask(uint8_t* mask, int64_t n, float p, uint64_t seed, void* stream);
int xt_dropout_add_fwd(const void* h, const void* a, void* out, int64_t n, float p,
                       uint64_t seed, int training, int dt, void* stream);

enum { XT_NORM_RMS = 0, XT_NORM_LN = 1 };  /* norm kinds (also the block stack's norm field) */

/* ---------------------------------------------------------------------------------
 * The residual path's dropout fused with its neighbouring pre-norm ([DO] § dropout 接在哪
 * (wiring): every residual add of the block is followed by the next sub-block's norm, and
 * every norm backward by the preceding site's dropout backward).  Same masks, same
 * arithmetic, same results as the separate calls, one pass over the rows:
 *   xt_dropout_add_norm_fwd: sum = h + dropout(a) over [rows, cols] (flat index i = r·cols + c,
 *     as xt_dropout_add_fwd), then y = norm(sum as stored) with its statistics:
 *     norm = XT_NORM_RMS: stat0 = inv_rms (xt_rms_norm_fwd; beta, stat1 unused);
 *     norm = XT_NORM_LN:  stat0 = mean, stat1 = rstd (xt_layernorm_fwd).
 *   xt_norm_bwd_dropout: the norm backward (xt_rms_norm_bwd with stat0 = inv_rms, or
 *     xt_layernorm_bwd with stat0 = mean, stat1 = rstd; dx required) that also writes
 *     g = dropout_bwd(dx as stored) (xt_dropout_bwd_ex from dx to g), g of dtype dt.
 * ------------------------------------------------------------------------------- */
int xt_dropout_add_norm_fwd(const void* h, const void* a, void* sum, const void* gamma,
                            const void* beta, void* y, float* stat0, float* stat1, int64_t rows,
                            int64_t cols, float p, uint64_t seed, int training, int norm, float eps,
                            int dt, void* stream);
int xt_norm_bwd_dropout(int norm, const void* d, const void* x, const void* gamma, const float* stat0,
                        const float* stat1, void* dx, void* dgamma, void* dbeta, void* g, int64_t rows,
                        int64_t cols, int dt, int dt_dx, int dt_param, void* ws, int acc_dx,
                        int acc_param, float p, uint64_t seed, int training, void* stream);

/* ---------------------------------------------------------------------------------
 * Embedding ([BP] § kernel-pair table k_embed_fwd/bwd; § Var gradienter lever i minnet):
 * h[t] = E[ids[t]] (+ P[t mod S] when P != NULL).  Backward: dE[v] = Σ_{t: ids[t]=v} dh[t]
 * summed in ascending t (deterministic), dP[s] = Σ_b dh[b·S+s].  With acc == 0 the rows
 * of dE that no token touches are zeroed.  T ≤ 16384.  The workspace (kept for the
 * interface) may be NULL.
 * ------------------------------------------------------------------------------- */
int xt_embedding_workspace_size(int64_t T, size_t* bytes);
int xt_embedding_fwd(const int32_t* ids, const void* E, const void* P, void* h, int64_t T, int S,
                     int64_t d, int64_t V, int dt, void* stream);
int xt_embedding_bwd(const int32_t* ids, const void* dh, void* dE, void* dP, int64_t T, int S,
                     int64_t d, int64_t V, int dt_dh, int dt_grad, void* ws, int acc,
                     void* stream);

/* ---------------------------------------------------------------------------------
 * Matmul on the tensor cores ([AE] op table row matmul: C = A@B; dA = d@Bᵀ, dB = Aᵀ@d).
 *   op(A) is M×K: trans_a = 0 ⇒ A stored [M, K] (ld lda); 1 ⇒ A stored [K, M].
 *   op(B) is K×N: trans_b = 0 ⇒ B stored [K, N] (ld ldb); 1 ⇒ B stored [N, K].
 *   C [M, N] (ld ldc) = alpha·op(A)@op(B)  (+ C when accumulate).
 * Two batch levels (outer × inner) with element strides, e.g. (batch, head) for attention.
 * dtype_ab: XT_BF16 (bf16 products) or XT_F32 (tf32 products); dtype_c: XT_F32 or XT_BF16.
 * Requirements (else XT_ERR_ALIGNMENT): A, B 16-byte aligned; lda, ldb and the A/B batch
 * strides are multiples of 16 bytes; C 16-byte aligned and ldc a multiple of 16 bytes.
 * causal (square attention blocks, 128-row granularity): 0 none; 1 skip output tiles
 * entirely above the diagonal block (n0 ≥ m0+128); 2 stop the K loop at m0+128 (A is a
 * causal probability block); 3 start the K loop at m0 (A is a transposed causal block).
 * ------------------------------------------------------------------------------- */
typedef struct xt_matmul_desc {
  int32_t M, N, K;
  int32_t trans_a, trans_b;
  int32_t batch_outer, batch_inner;
  int32_t dtype_ab, dtype_c;
  int32_t accumulate;
  int32_t causal;
  float alpha;
  int64_t lda, ldb, ldc;
  int64_t stride_a_outer, stride_a_inner;
  int64_t stride_b_outer, stride_b_inner;
  int64_t stride_c_outer, stride_c_inner;
} xt_matmul_desc;

/* Scratch bytes the call needs, laid out as
 *   [4096 bytes of stream-K flag words][tf32 staging][partial tiles]:
 *   - flag words: zero before the workspace's first use (e.g. cudaMemset once when it is
 *     allocated); each call leaves them zero.  A stream-K launch's CTAs signal through them
 *     that a partial tile is ready, so two matmul calls must not share a workspace while
 *     both can run (on two streams);
 *   - staging: XT_F32 operands read MN-major (trans_a = 1 or trans_b = 0) are first copied,
 *     transposed, into K-major scratch because the tf32 MMA is fed K-major operands only;
 *   - partial tiles: fp32 partial accumulators of a K split or of the stream-K schedule.
 * The schedule is chosen per problem from a per-tile time model: whole output tiles over
 * persistent CTAs, or (with a workspace, non-causal) a K split reduced in a fixed order by a
 * second kernel, or stream-K: every SM's CTA an equal share of the tiles' k-block
 * iterations, or tiles × s CTAs each computing one K slice of one tile; a tile shared by
 * several CTAs is summed, in CTA order, by the CTA holding its first k-blocks.  All are
 * deterministic.  ws = NULL (or fewer bytes than reported) restricts the choice
 * to whole tiles, and is an error for the tf32 staging case. */
int xt_matmul_workspace_size(const xt_matmul_desc* desc, size_t* bytes);
/* Schedule override for every later matmul call of the process (tests, tuning): 0 the
 * time model's choice (default), 1 whole tiles only, 2 a K split wherever one is allowed,
 * 3 stream-K over every SM wherever allowed, 4 stream-K in lockstep K slices (tiles × s
 * CTAs, each one K slice of one tile) wherever allowed.  XT_ERR_INVALID_ARG otherwise. */
int xt_gemm_set_schedule(int mode);
/* Process-wide override of the paired-CTA GEMM (bf16 operands, no causal mode, no GELU
 * epilogue): two CTAs of a cluster compute one 256-row tile with the paired tensor-core MMA,
 * each staging its own 128 rows of A and half of B's rows.  Its multicast form runs clusters
 * of two such pairs on vertically adjacent 256 × 256 tiles (whole tiles, an even number of
 * 256-row tiles), each CTA loading half of its B rows for both pairs.  0 = the time model's
 * choice (default; never the multicast form, which measured slower than the plain pairs on
 * the 12-layer stack's shapes), 1 = never, 2 = the plain pairs wherever allowed, 3 = the
 * multicast form wherever allowed (else as 2).  Every kernel accumulates in fp32 over the same K order; the
 * choice is deterministic for a given shape.  XT_ERR_INVALID_ARG otherwise. */
int xt_gemm_set_pairing(int mode);
/* Process-wide override of the GEMM tile width: 0 = the time model's choice (default), else
 * BN ∈ {64, 128, 192, 256} wherever it is a candidate for the problem (the model's choice
 * otherwise).  For measurement and tests.  XT_ERR_INVALID_ARG for other values. */
int xt_gemm_set_tile(int bn);
int xt_matmul_fwd(const xt_matmul_desc* desc, const void* A, const void* B, void* C, void* ws,
                  size_t ws_bytes, void* stream);
/* Backward of C = alpha·op(A)@op(B) given dC (layout of C, dtype dtype_ab):
 * dA = alpha·dC@op(B)ᵀ into A's layout, dB = alpha·op(A)ᵀ@dC into B's layout; dA/dB have
 * dtype dt_grad_a / dt_grad_b; either may be NULL.  causal must be 0. */
/* The GELU of the MLP ([BP] § Framåtgåendet: the up projection followed by exact GELU) fused
 * into the GEMM epilogue, gelu(a) = a·Φ(a):
 *   xt_matmul_gelu_fwd: C = alpha·op(A)@op(B) (the pre-activation, rounded to bf16) and
 *                       Y = gelu(C) evaluated on that rounded value;
 *   xt_matmul_gelu_bwd: C = (alpha·op(A)@op(B)) ∘ gelu'(X) with gelu'(a) = Φ(a) + a·φ(a),
 *                       X the saved pre-activation (the GELU backward applied to the product).
 * Y and X are bf16 with C's layout (ldc).  Restrictions (else XT_ERR_UNSUPPORTED /
 * XT_ERR_INVALID_ARG): dtype_ab = dtype_c = XT_BF16, one batch, accumulate = 0, causal = 0,
 * N a multiple of 64; Y / X 16-byte aligned.  Workspace as xt_matmul_workspace_size. */
int xt_matmul_gelu_fwd(const xt_matmul_desc* desc, const void* A, const void* B, void* C, void* Y,
                       void* ws, size_t ws_bytes, void* stream);
int xt_matmul_gelu_bwd(const xt_matmul_desc* desc, const void* A, const void* B, const void* X, void* C,
                       void* ws, size_t ws_bytes, void* stream);

int xt_matmul_bwd_workspace_size(const xt_matmul_desc* desc, size_t* bytes);
int xt_matmul_bwd(const xt_matmul_desc* desc, const void* A, const void* B, const void* dC,
                  void* dA, void* dB, int dt_grad_a, int dt_grad_b, int acc_a, int acc_b,
                  void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------------
 * FP8 E4M3 ([BP] § Vad generiska ramverk kostar, item 4: an FP8 E4M3 tensor-core path in the
 * mixed-precision pipeline; the pages give no format details, so the OCP E4M3 format is used:
 * bias 7, 3 mantissa bits, subnormals m·2⁻⁹, largest finite 448, no infinities).
 *   xt_quantize_fp8: per-tensor quantization of n elements of x (XT_F32 / XT_BF16):
 *     scale = 448 / max|x| (one float32 division; 1 when all are 0), out[i] = e4m3(x[i]·scale)
 *     rounded to nearest even and saturated to ±448; *dequant (device float) = max|x| / 448
 *     (1 when all are 0), the factor a code is multiplied by to stand for x.  The workspace
 *     (xt_quantize_fp8_workspace_size) holds per-block maxima.  Deterministic.
 *   xt_matmul_fp8_fwd: C [M, N] (+)= alpha · (*scale_a) · (*scale_b) · A Bᵀ on the tensor cores
 *     (tcgen05 kind::f8f6f4, float32 accumulation): A [M, K] and B [N, K] e4m3 codes with K
 *     contiguous (rows lda / ldb bytes apart, multiples of 16), C float32 or bf16 (ldc
 *     elements); scale_a / scale_b are device floats (may be NULL: 1), e.g. the dequant factors
 *     of xt_quantize_fp8.  A, B, C 16-byte aligned (else XT_ERR_ALIGNMENT).
 * ------------------------------------------------------------------------------- */
int xt_quantize_fp8_workspace_size(int64_t n, size_t* bytes);
int xt_quantize_fp8(const void* x, int64_t n, int dt, uint8_t* out, float* dequant, void* ws, size_t ws_bytes,
                    void* stream);
int xt_matmul_fp8_fwd(int64_t M, int64_t N, int64_t K, const uint8_t* A, int64_t lda, const uint8_t* B, int64_t ldb,
                      void* C, int64_t ldc, int dt_c, float alpha, const float* scale_a, const float* scale_b,
                      int accumulate, void* stream);

/* ---------------------------------------------------------------------------------
 * Optimizer step after the backward ([BP] § Ackumulation över mikrobatcher: gradients of
 * every microbatch are summed into the buffers, then scaled by 1/n_microbatches before one
 * optimizer step; [BP] § Parningsdisciplinen: gradient clipping as a partial and a final
 * gradient-norm reduction and a gradient scale; [BP] § Optimiser-tillståndet: AdamW with a
 * first moment m and a second moment v per weight).  Over n tensors i, all float32:
 *   s    = grad_scale (e.g. 1 / n_microbatches),  norm = ‖s·g‖₂ over every element of every
 *          tensor,  c = min(1, max_grad_norm / (norm + 1e-6))  (c = 1 when max_grad_norm ≤ 0),
 *   g'   = s·c·g,   m ← β₁ m + (1−β₁) g',   v ← β₂ v + (1−β₂) g'²,
 *   θ    ← θ (1 − lr·λ) − lr · (m / (1−β₁ᵗ)) / (√(v / (1−β₂ᵗ)) + ε)   (t = step ≥ 1).
 * param, m, v are updated in place; grad is read only.  shadow (NULL, or per tensor NULL or
 * a device pointer) receives the updated θ converted to shadow_dtype (XT_BF16 / XT_F32): the
 * working copy a bf16 model computes with while param holds the float32 master weights.
 * param, grad, m, v, shadow and numel are HOST arrays of n entries (device pointers, sizes).
 * norm_out (device float, may be NULL) receives norm.  The workspace
 * (xt_adamw_workspace_size) holds one partial sum per 4096-element tile and is needed when
 * clipping or norm_out is requested.  Deterministic: fixed-order sums, no atomics.
 * ------------------------------------------------------------------------------- */
typedef struct xt_adamw_config {
  float lr, beta1, beta2, eps, weight_decay;
  float max_grad_norm; /* ≤ 0: no clipping */
  float grad_scale;    /* applied to every gradient before the norm (1 / n_microbatches) */
  int32_t step;        /* t ≥ 1, for the bias corrections */
} xt_adamw_config;

int xt_adamw_workspace_size(int n, const int64_t* numel, size_t* bytes);
int xt_adamw_step(const xt_adamw_config* cfg, int n, float* const* param, const float* const* grad, float* const* m,
                  float* const* v, void* const* shadow, int shadow_dtype, const int64_t* numel, float* norm_out,
                  void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------------
 * Native block stack ([BP] § Framåtgåendet; [DO] § dropout 接在哪（wiring）):
 *   h = E[ids] (+ P);  per layer l:  h += dropout(attn(norm1 h), seed ⊕ l ⊕ 0xA77),
 *                                    h += dropout(mlp(norm2 h),  seed ⊕ l ⊕ 0xF70);
 *   logits = norm_f(h) @ Eᵀ;  loss = cross_entropy(logits, targets).
 * attn: q,k,v = x@W_qkv (W_qkv = [W_Q | W_K | W_V], [d, 3d]); optional RoPE on q, k;
 * per (b, head) P = softmax_causal(q kᵀ/√hd), o = P v; attn = o @ W_O.
 * mlp: SWIGLU: (silu(x@W_g) ∘ x@W_u) @ W_d with W_gu = [W_g | W_u] ([d, 2F]);
 *      GELU:   gelu(x@W_1) @ W_2.
 * xt_block_fwd runs the forward and keeps the saved tensors in ws; xt_block_bwd then adds
 * every parameter gradient into the grad buffers (+=, [BP] § Ackumulation över mikrobatcher);
 * call xt_block_zero_grads first for a fresh step.  No host synchronisation; the pair can
 * be captured in a CUDA graph.  xt_block_bwd runs the weight-gradient GEMMs on a second
 * stream of the device (created by the first xt_block_workspace_size call, never destroyed),
 * forked from and joined back into `stream` with events, so the work it enqueues is complete
 * when `stream` reaches its end; calls on one device must not be issued concurrently from
 * several host threads (they share that stream's events).  With recompute = 1 everything
 * stays on `stream`.
 * ------------------------------------------------------------------------------- */
enum { XT_MLP_SWIGLU = 0, XT_MLP_GELU = 1 };
/* Attention path: AUTO runs the fused kernels (xt_attention_*) when dtype is XT_BF16, hd is
 * 64 and d is a multiple of 8, else the composition of causal-tile GEMMs around the row
 * softmax (which also saves P [B, H, S, S]); COMPOSED forces the latter; FUSED requires the
 * former (XT_ERR_UNSUPPORTED otherwise). */
enum { XT_ATTN_AUTO = 0, XT_ATTN_COMPOSED = 1, XT_ATTN_FUSED = 2 };

typedef struct xt_block_config {
  int32_t B, S, d, H, hd, F, V, n_layers;
  int32_t norm;       /* XT_NORM_RMS or XT_NORM_LN */
  int32_t mlp;        /* XT_MLP_SWIGLU or XT_MLP_GELU */
  int32_t rope;       /* 1: rotate q and k */
  int32_t learned_pos;/* 1: P [S, d] added to the embedding */
  int32_t causal;     /* must be 1 */
  int32_t training;   /* 0: dropout is the identity */
  int32_t dtype;      /* activation and weight storage: XT_F32 or XT_BF16 */
  int32_t grad_dtype; /* parameter-gradient storage: XT_F32 or XT_BF16 */
  float eps;
  float p;            /* residual dropout probability */
  double rope_base;
  uint64_t base_seed;
  int32_t attention;  /* XT_ATTN_AUTO, XT_ATTN_COMPOSED or XT_ATTN_FUSED */
  int32_t recompute;  /* 1: activation recompute — the workspace keeps each layer's input only
                         and the backward recomputes the layer's forward (norm, projections,
                         attention, activation) from it before its backward; the recomputed
                         values are the forward's bit for bit (same kernels, same inputs,
                         counter-based dropout), so are the gradients; 0: keep everything */
} xt_block_config;

/* Per-layer parameter (and gradient) pointers; arrays of n_layers device pointers,
 * held in HOST memory.  Fields unused by the configuration may be NULL. */
typedef struct xt_block_params {
  const void* E;      /* [V, d] */
  const void* P;      /* [S, d] or NULL */
  const void* const* g1; const void* const* b1;
  const void* const* Wqkv; const void* const* Wo;
  const void* const* g2; const void* const* b2;
  const void* const* W_up;   /* [d, 2F] (SWIGLU) or [d, F] (GELU) */
  const void* const* W_down; /* [F, d] */
  const void* gf; const void* bf;
  void* dE; void* dP;
  void* const* dg1; void* const* db1;
  void* const* dWqkv; void* const* dWo;
  void* const* dg2; void* const* db2;
  void* const* dW_up; void* const* dW_down;
  void* dgf; void* dbf;
} xt_block_params;

/* The workspace holds the saved activations and every scratch buffer of the step; its first
 * 4096 bytes (the matmul scratch's stream-K flag words) must be zero before its first use. */
int xt_block_workspace_size(const xt_block_config* cfg, size_t* bytes);
int xt_block_fwd(const xt_block_config* cfg, const xt_block_params* prm, const int32_t* ids,
                 const int32_t* targets, float* loss, void* ws, void* stream);
int xt_block_bwd(const xt_block_config* cfg, const xt_block_params* prm, const int32_t* ids,
                 const int32_t* targets, void* ws, void* stream);
int xt_block_zero_grads(const xt_block_config* cfg, const xt_block_params* prm, void* stream);
/* Process-wide: 1 (default) the backward's weight-gradient GEMMs run on the second stream; 0 all
 * on `stream` (for measurement: a GEMM launch timed beside other kernels includes the time it
 * waits for SMs they hold).  Applies to backward calls enqueued afterwards; XT_ERR_INVALID_ARG
 * for other values. */
int xt_block_set_overlap(int on);

#ifdef __cplusplus
}
#endif
#endif /* XT_H */
