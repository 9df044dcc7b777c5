/*
 * lora_gb300.h -- C ABI of the GB300 (sm_103a) LoRA block-projection library.
 *
 * What is computed
 * ----------------
 * A LoRA linear with frozen base weight W [out x in] and adapter A [r x in],
 * B [out x r], scale s:
 *
 *     y = x W^T + s (x A^T) B^T                                               (1)
 *
 * ("Model Patches and Kernels", opake user guide, section "Fused LoRA operations",
 * row opake_lora_w: x @ W.T + x @ A @ B * s, written here in the PEFT layout with
 * A stored [r x in] and B stored [out x r]; s = alpha / r.)
 *
 * The gated MLP (same section, row opake_lora_mlp: gate + up + activation + down in
 * one call; activations from the same page, "Activation functions" table):
 *
 *     g = (1) with gate,  u = (1) with up,  h = act(g) * u,  y = (1) of h with down
 *     act = silu (SwiGLU), or GELU (GeGLU): exact (erf) or its tanh approximation
 *
 * The attention projections (row opake_lora_qkv: q, k, v share the input x; the
 * axolotl "monkeypatch.lora_kernels" reference, original_apply_qkv returning
 * (query, key, value) and original_apply_o for the output projection): q, k, v and
 * o are each (1); o's input is the attention output, which this library does not
 * compute.
 *
 * Backward computes the gradient of <dy, y> with respect to x and every A and B.
 * W is frozen and gets no gradient ("Model Patches and Kernels", section "Fused
 * linear cross-entropy": a frozen weight's gradient is skipped).  Adapters have no
 * dropout and no bias (axolotl apply_lora_kernel_patches note; MLP fusion is
 * bias-free per opake).
 *
 * Conventions (all entry points)
 * ------------------------------
 * - Tensors are bf16, row-major, dense (row stride = number of columns), in device
 *   memory, token-major for activations: x [M x in], y [M x out]; M = batch * seq.
 *   W [out x in], A [r x in], B [out x r], dA [r x in], dB [out x r].
 * - The caller owns and allocates every buffer, including `saved` and `ws`; the
 *   library allocates no memory and never synchronises (lora_poll_status and
 *   lora_trace_read aside).  All work is enqueued on `stream`, in order.  Kernels are
 *   launched with programmatic dependent launch (each waits for the previous work on
 *   the stream before it touches memory; environment LORA_PDL=0 turns the attribute
 *   off), so stream order holds as usual for the caller's own work around the calls.
 * - Gradient outputs (dx, dA, dB) are overwritten, not accumulated.
 * - Alignment: every pointer 16-byte aligned (`ws` and `saved` 256-byte aligned);
 *   every feature size (in, out, h, i, n_q, n_kv) a multiple of 8.  A and B need no
 *   alignment beyond their element size.  Violations return LORA_ERR_ALIGNMENT.
 * - Rank limits: 1 <= r, and (number of adapters sharing one input) * r <= 256,
 *   i.e. r <= 128 for the MLP's gate/up pair and r <= 85 for q/k/v; otherwise
 *   LORA_ERR_UNSUPPORTED.  Size limits: M and every feature size at most 2^31 - 1
 *   (32-bit row, column and tile indices); otherwise LORA_ERR_UNSUPPORTED.
 * - Every argument error returns before anything is enqueued.  No entry point
 *   aborts, throws or prints.
 * - `ws` must hold lora_*_workspace_bytes(...) bytes; its first 256 bytes hold the
 *   status word that kernels set asynchronously (zero them before first use;
 *   lora_poll_status reads and clears it).  `saved` must hold lora_*_saved_bytes(...)
 *   and is an opaque blob written by forward and read by backward.
 * - M == 0 is allowed: forward enqueues nothing, backward zero-fills dA and dB.
 * - Calls that share a `ws` must not overlap on the GPU (same stream is safe).
 */
#ifndef LORA_GB300_H
#define LORA_GB300_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  LORA_ACT_SWIGLU = 0,      /* silu(g) * u */
  LORA_ACT_GEGLU_TANH = 1,  /* gelu_tanh(g) * u, 0.5 g (1 + tanh(sqrt(2/pi)(g + 0.044715 g^3))) */
  LORA_ACT_GEGLU_ERF = 2    /* gelu(g) * u, 0.5 g (1 + erf(g / sqrt 2)) */
} lora_act_t;

typedef enum {
  LORA_OK = 0,
  LORA_ERR_INVALID_ARG = 1,   /* NULL pointer, negative size, bad enum, non-finite s */
  LORA_ERR_ALIGNMENT = 2,     /* pointer or feature size violates the alignment rules */
  LORA_ERR_UNSUPPORTED = 3,   /* rank or size beyond the limits above */
  LORA_ERR_WORKSPACE = 4,     /* ws_bytes below the workspace query */
  LORA_ERR_CUDA = 5,          /* a CUDA runtime call or kernel launch failed */
  LORA_ERR_TIMEOUT = 6,       /* a kernel's bounded wait expired (read by lora_poll_status) */
  LORA_ERR_DEVICE_INPUT = 7   /* a value in device memory was out of range: a RoPE position
                                 outside [0, n_pos) (read by lora_poll_status; position 0
                                 was used in its place) */
} lora_status_t;

/* One frozen base weight and its adapter: device pointers, bf16, row-major.
 * W [out x in], A [r x in], B [out x r]. */
typedef struct {
  const void* W;
  const void* A;
  const void* B;
} lora_linear_t;

/* Gradient outputs of one adapter: dA [r x in], dB [out x r], bf16, overwritten. */
typedef struct {
  void* dA;
  void* dB;
} lora_grads_t;

/* ---------------------------------------------------------------- single linear
 * (1) for one projection ("opake_lora_w").  saved holds the rank-r projection x A^T
 * and the adapter packed for backward; pass NULL for inference. */
size_t lora_linear_saved_bytes(int64_t M, int64_t in, int64_t out, int r);
size_t lora_linear_workspace_bytes(int64_t M, int64_t in, int64_t out, int r);
lora_status_t lora_linear_forward(int64_t M, int64_t in, int64_t out, int r, float s,
                                  const void* x, lora_linear_t lin, void* y, void* saved,
                                  void* ws, size_t ws_bytes, cudaStream_t stream);
/* dx [M x in] = dy W + s (dy B) A;  dA = s (dy B)^T x;  dB = s dy^T (x A^T).
 * x is the forward input again; saved is what forward wrote, including the adapter
 * packed as this call's operands (with the forward's s): lin must be the forward's
 * (its W is read here, its A and B only checked), and s the same, as autograd uses the
 * tensors a forward saved. */
lora_status_t lora_linear_backward(int64_t M, int64_t in, int64_t out, int r, float s,
                                   const void* x, lora_linear_t lin, const void* saved,
                                   const void* dy, void* dx, lora_grads_t grads,
                                   void* ws, size_t ws_bytes, cudaStream_t stream);

/* Forward of the single linear (inference: nothing is saved) that allocates nothing
 * and takes no workspace.  The pages have no counterpart; it exists for callers that
 * cannot allocate device memory where they run this projection -- a plugin inside a
 * host framework that owns all device memory and passes the plugin only its input and
 * output buffers, or a latency-critical loop that must never call cudaMalloc (which
 * can synchronise the device).  Scratch comes from a fixed 32 MiB array inside the
 * library, which every GPU that loads the library holds until the process exits.
 * - Problems whose forward needs more than 32 MiB of scratch (the forward's share of
 *   lora_linear_workspace_bytes(M, in, out, r), which also counts the backward's) are
 *   rejected with LORA_ERR_WORKSPACE before anything is enqueued; other argument rules
 *   are those of lora_linear_forward with saved == NULL, and so is the result, up to
 *   the order of the f32 sums (this call always gives each 256 x 256 output tile to
 *   one CTA pair).
 * - Asynchronous errors (an expired bounded wait) set the status word at the front of
 *   the array; lora_poll_status(NULL, stream) reads and clears it.  It stays set across
 *   calls until polled.
 * - The first call on a device, and the first after the device's context was
 *   destroyed and created again (cudaDeviceReset), looks up the array's device address;
 *   make that first call before any stream capture.
 * - Every call on a device shares the one array and leaves its contents behind; calls
 *   whose GPU work overlaps (other streams, other threads) race and corrupt each
 *   other's results.  Calls in order on one stream are safe. */
lora_status_t lora_linear_forward_noalloc(int64_t M, int64_t in, int64_t out, int r, float s,
                                          const void* x, lora_linear_t lin, void* y,
                                          cudaStream_t stream);

/* ---------------------------------------------------------------- gated MLP
 * x [M x h] -> y [M x h] through gate/up [i x h] and down [h x i] ("opake_lora_mlp").
 * saved (NULL for inference) receives g, u, h and the rank-r projections for
 * backward (x [A_g; A_u]^T also transposed, for the backward's single pass over dg, du
 * when r <= 16), and the adapters packed as the backward's operands. */
size_t lora_mlp_saved_bytes(int64_t M, int64_t h, int64_t i, int r);
size_t lora_mlp_workspace_bytes(int64_t M, int64_t h, int64_t i, int r);
lora_status_t lora_mlp_forward(int64_t M, int64_t h, int64_t i, int r, float s, lora_act_t act,
                               const void* x, lora_linear_t gate, lora_linear_t up,
                               lora_linear_t down, void* y, void* saved,
                               void* ws, size_t ws_bytes, cudaStream_t stream);
/* Gradients of <dy, y>: dx [M x h] and dA/dB of gate, up and down.  Needs the
 * forward's x and saved blob (the activation and its derivative are recomputed from
 * the saved g, u).  The adapters enter as the forward packed them into saved (with its
 * s), as autograd uses the tensors a forward saved: gate, up and down must be the
 * forward's (their W is read here; their A and B only checked), and s the same. */
lora_status_t lora_mlp_backward(int64_t M, int64_t h, int64_t i, int r, float s, lora_act_t act,
                                const void* x, lora_linear_t gate, lora_linear_t up,
                                lora_linear_t down, const void* saved, const void* dy,
                                void* dx, lora_grads_t d_gate, lora_grads_t d_up,
                                lora_grads_t d_down, void* ws, size_t ws_bytes,
                                cudaStream_t stream);

/* Per-example adapter gradients, for DP-SGD (the opake use case: per-example
 * gradients by vmap(grad) before clipping; "Model Patches and Kernels").  The M tokens
 * are n_examples examples of seq = M / n_examples consecutive tokens (M must be a
 * multiple of n_examples; token t belongs to example t / seq).  Writes dx as
 * lora_mlp_backward does, and for each adapter the gradient of every example on its
 * own: d_*.dA [n_examples x r x in], d_*.dB [n_examples x out x r] (bf16, example-major).
 * sq_norms (NULL or float [n_examples]) receives each example's squared L2 norm over
 * all six adapter gradients, summed from the bf16 results in a fixed order.  ws must
 * hold lora_mlp_per_example_workspace_bytes(M, h, i, r, n_examples). */
size_t lora_mlp_per_example_workspace_bytes(int64_t M, int64_t h, int64_t i, int r, int64_t n_examples);
lora_status_t lora_mlp_backward_per_example(int64_t M, int64_t h, int64_t i, int r, float s, lora_act_t act,
                                            int64_t n_examples, const void* x, lora_linear_t gate,
                                            lora_linear_t up, lora_linear_t down, const void* saved,
                                            const void* dy, void* dx, lora_grads_t d_gate,
                                            lora_grads_t d_up, lora_grads_t d_down, float* sq_norms,
                                            void* ws, size_t ws_bytes, cudaStream_t stream);

/* Rotary position embedding of q and k ("Model Patches and Kernels", section "Rotary
 * position embeddings (RoPE)": q and k rotated together, GQA head counts; RoFormer's
 * position encoding).  Every head (head_dim features) of q and k is rotated pair by
 * pair, the pair being features (c, c + head_dim/2) of the head:
 *   q'[c] = q[c] cos - q[c + d/2] sin,  q'[c + d/2] = q[c + d/2] cos + q[c] sin,
 * with cos, sin = cos[pos[m]][c], sin[pos[m]][c] for token m.  The tables are the
 * caller's (lora_rope_table fills RoFormer's p * base^(-2c/d); scaled variants are
 * any other table).  Device pointers: cos, sin f32 [n_pos x head_dim/2] row-major,
 * 16-byte aligned; pos int32 [M], 4-byte aligned.  head_dim is 64, 128 or 256 and
 * divides n_q and n_kv.  A position outside [0, n_pos) is read as 0 and reported by
 * lora_poll_status as LORA_ERR_DEVICE_INPUT. */
typedef struct {
  const float* cos;
  const float* sin;
  const int32_t* pos;
  int64_t n_pos;
  int head_dim;
} lora_rope_t;

/* Fills cos/sin [n_pos x head_dim/2] (f32, device, 16-byte aligned) with the cosine
 * and sine of p * base^(-2c/head_dim), computed in double and rounded once.
 * head_dim even and >= 2, n_pos >= 1, base > 0, else LORA_ERR_INVALID_ARG. */
lora_status_t lora_rope_table(float* cos, float* sin, int64_t n_pos, int head_dim, double base,
                              cudaStream_t stream);

/* ---------------------------------------------------------------- Q/K/V + O
 * q = (1)(x; q) [M x n_q], k, v = (1)(x; k or v) [M x n_kv] ("opake_lora_qkv"), and
 * yo = (1)(o_in; o) [M x h] with W_o [h x n_q] ("original_apply_o").  Attention runs
 * between the two halves in a real block, so either half may be skipped: x == NULL
 * skips q/k/v, o_in == NULL skips O.  bias_qkv is NULL or the frozen base-layer
 * biases of q, k and v, bf16 [n_q + 2 n_kv] (q's, then k's, then v's), 16-byte
 * aligned, added to q, k, v ("Fused LoRA operations": QKV fusion supports optional
 * frozen base-layer biases); a frozen bias gets no gradient, so backward does not
 * take it.  rope is NULL or the rotary embedding applied to q and k after the bias,
 * in the projection's epilogue (lora_rope_t above; ignored when x == NULL).  saved
 * (NULL for inference) receives the rank-r projections (also transposed where the
 * backward's single passes read them) and the adapters packed for backward. */
size_t lora_qkvo_saved_bytes(int64_t M, int64_t h, int64_t n_q, int64_t n_kv, int r);
size_t lora_qkvo_workspace_bytes(int64_t M, int64_t h, int64_t n_q, int64_t n_kv, int r);
lora_status_t lora_qkvo_forward(int64_t M, int64_t h, int64_t n_q, int64_t n_kv, int r, float s,
                                const void* x, lora_linear_t q, lora_linear_t k,
                                lora_linear_t v, void* yq, void* yk, void* yv,
                                const void* o_in, lora_linear_t o, void* yo,
                                const void* bias_qkv, const lora_rope_t* rope, void* saved,
                                void* ws, size_t ws_bytes, cudaStream_t stream);
/* Gradients of <dyq, q> + <dyk, k> + <dyv, v> (dx = their sum over the three
 * projections, and dA/dB of q, k, v) and of <dyo, yo> (do_in and dA/dB of o).
 * x == NULL skips the q/k/v half, o_in == NULL the O half.  With rope (the one the
 * forward used), dyq and dyk are gradients of the rotated q and k: they are turned
 * back by the transpose rotation (into the workspace) before the projections'
 * backward.  The adapters enter as the forward packed them into saved (with its s):
 * q, k, v, o must be the forward's (their W is read here; their A and B only
 * checked), and s the same. */
lora_status_t lora_qkvo_backward(int64_t M, int64_t h, int64_t n_q, int64_t n_kv, int r, float s,
                                 const void* x, lora_linear_t q, lora_linear_t k,
                                 lora_linear_t v, const void* o_in, lora_linear_t o,
                                 const void* saved, const lora_rope_t* rope,
                                 const void* dyq, const void* dyk,
                                 const void* dyv, void* dx, const void* dyo, void* do_in,
                                 lora_grads_t d_q, lora_grads_t d_k, lora_grads_t d_v,
                                 lora_grads_t d_o, void* ws, size_t ws_bytes,
                                 cudaStream_t stream);

/* ---------------------------------------------------------------- status, counters
 * lora_poll_status: synchronises `stream`, reads the asynchronous status word in
 * ws, clears it, and returns LORA_OK, LORA_ERR_TIMEOUT or LORA_ERR_DEVICE_INPUT
 * (timeout first when both are set; LORA_ERR_CUDA if the synchronisation itself
 * fails).  ws == NULL reads and clears the status word of the current device's
 * lora_linear_forward_noalloc scratch instead (the word that call's kernels set). */
lora_status_t lora_poll_status(void* ws, cudaStream_t stream);
const char* lora_status_string(lora_status_t status);
/* Kernels this library has launched in this process (all entry points). */
uint64_t lora_launch_count(void);

/* ---------------------------------------------------------------- bounded waits
 * Every wait inside the GEMM kernels (a pipeline stage, an accumulator buffer) is
 * bounded.  When one runs out, the kernel stops issuing work, lets its own copies and
 * MMAs in flight finish, frees its tensor memory and exits; the status word in `ws`
 * then reads LORA_ERR_TIMEOUT (see lora_poll_status) and that call's outputs are
 * undefined.  The CUDA context stays usable.  The pages define no such mechanism.
 *
 * lora_set_wait_timeout: the limit in nanoseconds for launches enqueued after the
 * call, process-wide (all devices, all threads).  0 restores the default of 2 s.
 * Accepted range 1 ms .. 60 s, else LORA_ERR_INVALID_ARG.  A limit shorter than
 * the slowest tile of a workload (tens of microseconds for the shapes here, longer
 * when the GPU is time-sliced with other processes) makes healthy calls fail.
 * The limit is wall-clock time (the GPU's nanosecond timer), whatever the SM clock.
 * lora_wait_timeout: the current limit in nanoseconds. */
lora_status_t lora_set_wait_timeout(uint64_t ns);
uint64_t lora_wait_timeout(void);

/* ---------------------------------------------------------------- split tail
 * The projection GEMMs deal whole 256 x 256 output tiles round-robin to pairs of SMs.
 * When the last wave would leave pairs idle, the tiles of that wave (all tiles, when
 * there are fewer than pairs) can each be cut into 2 to 4 equal k-ranges computed by
 * different pairs; the last piece of a tile to finish adds the others' f32 partial
 * sums, in a fixed order, before the epilogue, so results stay deterministic for a
 * given device and mode (and match the whole-tile schedule up to the order of the f32
 * sums).  The partial sums live in the call's workspace (the size queries include
 * them).  Not from the pages: a scheduling choice of this library.
 *
 * lora_set_split_tail: 0 (default) cuts the tail into the number of pieces (2 to 4)
 * for which a cost model of the partial sums expects the launch to gain most, if at
 * least 2%; 1 never cuts; 2, 3 or 4 cuts every tail into that many pieces whenever the
 * launch allows it (every group with the same k-extent, at least 8 k-blocks per tile
 * and two per piece, a tail of at most 128 tiles).  Process-wide, for launches enqueued
 * after the call; the environment variable LORA_SPLIT_TAIL=1..4 sets the initial mode.
 * Other values return LORA_ERR_INVALID_ARG.  lora_split_tail: the current mode. */
lora_status_t lora_set_split_tail(int mode);
int lora_split_tail(void);

/* Test hook for the failure path (no counterpart in the pages): the next `launches`
 * GEMM launches (0 .. 64; 0 cancels) each leave the first pipeline stage of every
 * CTA's first tile unfilled, so the waits on it expire after the wait limit and the
 * call reports LORA_ERR_TIMEOUT through the status word.  Nothing faults, traps or
 * hangs: the waits are the bounded ones above.  Returns LORA_ERR_INVALID_ARG out of
 * range. */
lora_status_t lora_test_expire_waits(int launches);

/* Launch tracing, for measurement.  lora_trace_enable(n) makes every later launch (of
 * the kinds lora_trace_kinds selects; all by default) record a pair of CUDA events
 * around itself on its stream, keeping the first n launches (0 disables and frees
 * the events).  lora_trace_read synchronises the
 * recorded events, fills kind[] and ms[] (kernel kinds below) for up to `max`
 * launches, and restarts the trace; it returns the number filled or -1 on error. */
enum {
  LORA_KIND_PACK = 0,        /* adapter packing */
  LORA_KIND_REDUCE = 1,      /* split-K sums of the rank-r products; per-example norms */
  LORA_KIND_RANK_PROJ = 2,   /* token-major rank-r projections (x A^T, dy B, dg B) */
  LORA_KIND_RANK_GRAD = 3,   /* reductions over tokens (dA, dB) */
  LORA_KIND_GATE_UP = 4,     /* gate/up GEMM with the activation epilogue */
  LORA_KIND_PROJ = 5,        /* plain projection GEMM (down, q/k/v, o) */
  LORA_KIND_ACT_BWD = 6,     /* dh GEMM with the activation-derivative epilogue */
  LORA_KIND_DGRAD = 7,       /* input-gradient GEMM (dx, d o_in) */
  LORA_KIND_ROPE = 8         /* RoPE transpose rotation of dy_q, dy_k; RoPE tables */
};
lora_status_t lora_trace_enable(int capacity);
int lora_trace_read(int* kind, float* ms, int max);
/* Restricts tracing to the kinds whose bit is set in mask (bit k: kind k; all by
 * default).  Events between two launches serialise them, so tracing only the kernel
 * being measured keeps the others' overlap (programmatic dependent launch) intact. */
void lora_trace_kinds(unsigned mask);

#ifdef __cplusplus
}
#endif

#endif /* LORA_GB300_H */
