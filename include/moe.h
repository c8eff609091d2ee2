/*
 * moe.h -- C ABI of the GB300 (sm_103a) single-GPU Mixture-of-Experts layer.
 *
 * The layer: router logits -> top-k expert selection -> token dispatch ->
 * per-expert SwiGLU FFN -> weighted combine, its backward pass, and a
 * small-batch decode path.
 *
 * What it follows. "Cursor открыл код ядра Mixture of Experts: обучение MoE
 * ускоряется до 2,37 раза" (dzen.guru), section "Что именно тормозило обучение
 * MoE-моделей?": every MoE layer routes each token to experts, runs the
 * experts, and gathers the results back; section "Три решения, которые дали
 * результат": receivers pull the tokens they need (pull dispatch), results are
 * pushed back (push combine), no CPU in the loop, no dropped tokens, a fixed
 * ring buffer walked in reverse in the backward pass, one deterministic GPU
 * call, BF16 and MXFP8. "Cursor a réécrit le décodage de MoE" (toolnavs.com),
 * sections "Cursor a réécrit le décodage de MoE" and "1.84x plus de vitesse
 * ...": small-batch decode where each warp owns one output value, the whole
 * layer in two kernels, output closer to an FP32 reference.
 * The pages give no formulas. The layer computed here:
 *   l = x Wr^T (fp32)                       key = l + b (fp32, selection only)
 *   idx[t, 0..k-1] = the k largest keys, largest first, ties to the lower expert
 *   gate: softmax of the selected logits (renorm) or of all E (taken at idx),
 *         or route_scale * sigmoid(l) / sum over selected (renorm) or without /sum
 *   y_t = shared(x_t) + sum_{j=0}^{k-1} gate[t, j] * FFN_{idx[t, j]}(x_t)
 *   FFN_e(x) = (silu(x Wg[e]^T) * (x Wu[e]^T)) Wd[e]^T, shared expert = slot E.
 *
 * Conventions for every call:
 *  - Pointers named "device" must be device memory; the caller owns all of it.
 *    The library never allocates device memory except one small array in
 *    moe_create (the status word and a few counters). Scratch comes from the
 *    caller's `workspace` (sizes from moe_workspace_size), 256-byte aligned.
 *  - Every compute call only enqueues work on `stream` (a cudaStream_t passed
 *    as void*; NULL = legacy default stream) and never synchronises the host
 *    (moe_backward forks part of its work to a stream of the handle and joins
 *    it back into `stream` with events).
 *  - Arguments are validated on the host first; a bad argument returns an
 *    error code and launches nothing. Launch failures return MOE_ERR_CUDA.
 *    Errors detected on the device (an index out of range, a pipeline wait
 *    that timed out) are written to the handle's device status word; read it
 *    with moe_get_status (the only call that synchronises).
 *  - Row-major layouts. "bf16" storage means IEEE bfloat16 (uint16 bit
 *    patterns); fp32 storage for the MOE_FP32 precision.
 *  - A handle may be used from one stream at a time.
 *  - Results are bit-identical between runs for identical inputs (no floating
 *    point atomics; every sum has a fixed order).
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct moe_handle_s* moe_handle;

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,   /* null pointer, size out of range, k > E, ... */
  MOE_ERR_UNSUPPORTED = 2,   /* valid request the library does not implement (shape multiple, precision) */
  MOE_ERR_WORKSPACE = 3,     /* workspace or context smaller than required / misaligned */
  MOE_ERR_CUDA = 4,          /* a CUDA runtime call failed */
  MOE_ERR_TIMEOUT = 5,       /* device status: a pipeline wait exceeded its limit */
  MOE_ERR_DEVICE_INDEX = 6,  /* device status: an index read on the device was out of range */
  MOE_ERR_NO_WEIGHTS = 7     /* compute call before moe_set_weights */
} moe_status;

typedef enum { MOE_ROUTER_SOFTMAX = 0, MOE_ROUTER_SIGMOID = 1 } moe_router_kind;
typedef enum { MOE_FP32 = 0, MOE_BF16 = 1, MOE_MXFP8 = 2 } moe_precision;

typedef struct {
  int T_max;          /* largest token count any call will pass */
  int d;              /* hidden size */
  int E;              /* routed experts, 1..256 */
  int n_shared;       /* shared experts: 0 or 1 (stored as expert slot E) */
  int f;              /* SwiGLU intermediate width */
  int k;              /* experts per token, 1..min(E, 8) */
  int router;         /* moe_router_kind */
  int renorm;         /* 1: renormalise gates over the k selected experts */
  float route_scale;  /* multiplies the routed gates (1 for a plain softmax router) */
  int prec;           /* moe_precision of activations, weights and outputs */
  int chunk_tokens;   /* tokens per chunk of moe_train_chunked (0: whole batch) */
  size_t ring_bytes;  /* informational: the ring size the caller intends to pass to moe_train_chunked */
} moe_config;

/* Create a handle for one layer shape on the current CUDA device. Validates
 * the config (MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED) and allocates one
 * small device array (the status word, the decode router's counter and the
 * fused kernels' counters: 4 x (T_max (k+S) / 128 + E + S + 72)
 * bytes, the library's only allocation); on the tensor-core paths (bf16 and
 * MXFP8) it also creates one stream and three events for side work
 * (moe_backward's router backward, moe_train_chunked's next-chunk routing). */
moe_status moe_create(const moe_config* cfg, moe_handle* out);
moe_status moe_destroy(moe_handle h);

/* Bytes the caller must provide, for T tokens (T <= T_max):
 *   fwd_ws:   workspace of moe_forward / moe_route / moe_decode
 *   ctx:      activations saved by a training forward for moe_backward
 *   bwd_ws:   workspace of moe_backward
 *   packed:   packed weight buffer of moe_set_weights (independent of T)
 * Any output pointer may be NULL. */
moe_status moe_workspace_size(moe_handle h, int T, size_t* fwd_ws, size_t* ctx, size_t* bwd_ws,
                              size_t* packed);

/* Pack the layer's weights (device pointers, storage type of cfg.prec; bf16
 * for MXFP8) into the caller-owned device buffer `packed`:
 *   Wr [E, d]   router weight           bias [E] fp32 selection bias (NULL: zeros)
 *   Wg [E+S, f, d], Wu [E+S, f, d]      gate / up projections, rows = outputs
 *   Wd [E+S, d, f]                      down projection
 * Enqueued on `stream`; the source buffers may be freed once it has run. The
 * handle keeps `packed` and uses it in every later call: it must stay
 * allocated and unmodified. */
moe_status moe_set_weights(moe_handle h, const void* Wr, const float* bias, const void* Wg,
                           const void* Wu, const void* Wd, void* packed, void* stream);

/* Route T tokens x [T, d] (device). Writes (device, caller-owned):
 *   idx [T, k] int32, gate [T, k] fp32, cnt [E] int32, off [E+1] int32 (exclusive
 *   prefix of cnt), perm [T*k] int32 (sorted position -> assignment t*k+j, sorted
 *   by (expert, assignment)), inv [T*k] int32 (perm^-1), logits [T, E] fp32.
 * logits_override (nullable, device [T, E] fp32): route these logits instead of
 * computing x Wr^T (x may then be NULL). Any output may be NULL except logits
 * when logits_override is NULL. Uses `workspace` (fwd_ws bytes). */
moe_status moe_route(moe_handle h, const void* x, int T, const float* logits_override,
                     float* logits, int32_t* idx, float* gate, int32_t* cnt, int32_t* off,
                     int32_t* perm, int32_t* inv, void* workspace, void* stream);

/* Forward: y [T, d] = layer(x [T, d]) (device, storage type of cfg.prec; bf16
 * for MXFP8). ctx (nullable): when given (ctx bytes), the routing and the
 * expert pre-activations are saved there for moe_backward (training); NULL for
 * inference. */
moe_status moe_forward(moe_handle h, const void* x, int T, void* y, void* ctx, void* workspace,
                       void* stream);

/* Backward of the forward that filled ctx with the same x and T. dy [T, d] is
 * dL/dy. Writes (not accumulates) dx [T, d], dWr [E, d] fp32, and dWg, dWu
 * [E+S, f, d], dWd [E+S, d, f] in the storage type (fp32 for MOE_FP32, else
 * bf16). The selection bias gets no gradient. On the bf16 tensor-core path the
 * router backward and the dx gather-sum run on a stream of the handle's own,
 * forked from and joined back into `stream` with events (so the call stays
 * asynchronous on `stream` and capturable in a CUDA graph); calls on one
 * handle must therefore come from one host thread at a time. */
moe_status moe_backward(moe_handle h, const void* x, const void* dy, int T, const void* ctx,
                        void* dx, float* dWr, void* dWg, void* dWu, void* dWd, void* workspace,
                        void* stream);

/* Chunked training step over a fixed ring of saved activations. The MoK page
 * ("Три решения, которые дали результат") processes tokens in compute batches
 * of at least 2368 tokens and keeps saved activations in a fixed ring buffer
 * of a few hundred MB, walked in reverse in the backward pass so that fewer
 * activations are replayed. Here: chunks of cfg.chunk_tokens tokens (the whole
 * batch when 0); the forward of chunk c saves its routing and expert
 * pre-activations into ring slot c mod R, R = ring_bytes / slot_bytes; the
 * backward walks c = n-1 .. 0 and recomputes chunk c's forward only when a
 * later chunk overwrote its slot (c < n - R), i.e. n - R recomputes.
 * x, dy [T, d] in, y, dx [T, d] out (device, storage type of cfg.prec, bf16 for
 * MXFP8); dWr, dWg, dWu, dWd as in moe_backward, summed over chunks in backward
 * order (fp32 within a chunk, one bf16 rounding per chunk; dWr in fp32).
 * ring (device, >= slot_bytes, 256-byte aligned) and workspace (device,
 * workspace_bytes) come from moe_train_chunked_sizes. *recomputed (nullable,
 * host) receives the number of recomputed chunk forwards. With at least two
 * ring slots, the routing of chunk c + 1 (router GEMM, top-k, counts,
 * offsets, permutation) runs on the handle's own stream while chunk c's
 * expert GEMMs run (the page's "medium granularity" overlap, on one GPU),
 * forked from and joined back into `stream` with events, so the call stays
 * asynchronous on `stream` and capturable in a CUDA graph; results do not
 * depend on it. Asynchronous on `stream` like every compute call. */
moe_status moe_train_chunked_sizes(moe_handle h, int T, size_t* slot_bytes, size_t* workspace_bytes,
                                   int* n_chunks);
moe_status moe_train_chunked(moe_handle h, const void* x, const void* dy, int T, void* y, void* dx, float* dWr,
                             void* dWg, void* dWu, void* dWd, void* ring, size_t ring_bytes, void* workspace,
                             int* recomputed, void* stream);

/* Small-batch decode: y [B, d] bf16 = layer(x [B, d] bf16), 1 <= B <= 64,
 * cfg.prec MOE_BF16 or MOE_MXFP8 (MOE_FP32: MOE_ERR_UNSUPPORTED). Below the
 * crossover batch (moe_set_decode_crossover; default 4): warp-per-output
 * kernels with fp32 intermediates ("Cursor a réécrit le décodage de MoE",
 * toolnavs.com); from it, the grouped-GEMM forward. An MXFP8 layer decodes on
 * its E4M3 weights and computes its MXFP8 forward on the B tokens: x quantised
 * along d, h along f. workspace: fwd_ws of moe_workspace_size for T = B. */
moe_status moe_decode(moe_handle h, const void* x, int B, void* y, void* workspace, void* stream);

/* Batch size from which moe_decode runs the tensor-core grouped-GEMM forward
 * (moe_forward on the B tokens, inference) instead of the warp-per-output
 * kernels, on layers that have the tensor-core path (bf16 and MXFP8). On GB300
 * at DeepSeek-V3 shapes the warp kernels win at B = 1 and 2 and the grouped
 * GEMMs from B = 4 in both precisions (the warp kernels' per-token work grows
 * with B while the GEMMs read each used expert's weights once), so the default
 * is 4. b_min = 65 keeps every
 * batch on the warp kernels. Both paths compute the layer within the
 * precision's tolerance (the warp kernels keep h in fp32, the GEMM path rounds
 * it to the storage type, as moe_forward does). Host-only; b_min outside
 * 1..65 returns MOE_ERR_INVALID_ARG. */
moe_status moe_set_decode_crossover(moe_handle h, int b_min);

/* Tensor-core scheduling of the bf16 expert GEMMs (gate/up, down, dY.Wd, dx).
 * mode 1 runs them on pairs of SMs: 2-CTA clusters, one
 * tcgen05.mma.cta_group::2 per K step over a 256-row tile, each CTA holding
 * its own 128 rows and half of the weight tile. mode 0 runs one CTA per
 * 128-row tile. mode 2 runs one CTA per two 128-row tiles of an expert's
 * rows on one SM: two M = 128 MMAs per K step share each staged weight tile
 * (an expert's last, odd tile runs alone), so a pipeline stage carries twice
 * the MMA work. Modes 0 and 2 accumulate every output element with the same
 * instructions in the same K order, so their results are bit-identical; mode 1
 * agrees with them up to fp32 summation order. Each mode is deterministic.
 * Host-only; another mode returns MOE_ERR_INVALID_ARG. */
moe_status moe_set_pairs(moe_handle h, int mode);

/* Forward of a bf16 tensor-core layer as one persistent kernel, following the
 * one-call design of "Cursor открыл код ядра Mixture of Experts..." (section
 * "Три решения, которые дали результат"), on one GPU.
 * on = 1: the two expert GEMMs in one kernel: the gate/up GEMM (A5) and the
 * down GEMM (A6) run as one cooperative launch over a single tile order, a
 * down tile starting as soon as the gate/up tiles of its 128 rows have stored
 * h (per-row-block arrival counters held by the handle, waits bounded by the
 * device timeout), so no SM idles through the gate/up tail and the kernel
 * boundary; routing (A1-A4) and the combine (A7) stay separate launches.
 * on = 2: the whole forward in one cooperative launch: the router GEMM (the
 * same K splits as the separate launch, partials added in split order), top-k
 * and gates, chunk histograms, scan, permutation, the expert tiles taken from
 * a device tile queue (an atomic head; the dependency counters of on = 1),
 * and the combine, phases separated by grid-wide barriers; every wait is
 * bounded and past its limit records MOE_ERR_TIMEOUT and ends the call's work.
 * Results of both modes are bit-identical to on = 0 (the default, separate
 * launches). On GB300 mode 1 is 4-8% faster than separate launches on the
 * 2048-token layer at T <= 2048 and slower on the DeepSeek-V3 shape; mode 2
 * is faster than separate launches only at small T (T = 64), its routing and
 * combine phases running at one CTA per SM. Host-only. A nonzero value for a
 * layer without the bf16 tensor-core path returns MOE_ERR_UNSUPPORTED; other
 * values MOE_ERR_INVALID_ARG. While on != 0, calls on one handle must not run
 * concurrently on two streams (the counters are per handle). */
moe_status moe_set_fused(moe_handle h, int on);

/* Wait for the handle's queued work on `stream`, then read and clear the
 * device status word into *device_status (MOE_OK if no device error). */
moe_status moe_get_status(moe_handle h, void* stream, int* device_status);

/* Routing for callers that cannot allocate device memory: the same outputs
 * as moe_route with logits computed from x (logits, idx, gate, cnt, off, perm,
 * inv; all required, device, caller-owned), without a workspace argument. The
 * pages describe no such call; it exists for callers that may not allocate,
 * such as a plugin inside a host program that owns all device memory, or a
 * serving loop that bans cudaMalloc/cudaFree after start-up because they can
 * block and synchronise the device.
 * Its scratch is one fixed 4 MiB array inside the library, plus a 24 MiB one
 * for the split-K partials of the router GEMM (both held on every GPU that
 * loads the library until the process exits). A call needs
 *   2*pad(4*ceil(T*k/1024)*E) + 2*pad(4*(E+S+1)) + pad(24*(E+S+1))
 *   + 2*pad(4*T*(k+S)) bytes of the 4 MiB,
 * pad() rounding up to 256; larger T returns MOE_ERR_WORKSPACE before any
 * launch (E = 256, k = 8, S = 1 allows T up to 47,544 tokens).
 * The first call on a device looks up the array's address there; make that
 * first call before any stream capture. The address is kept for the life of
 * the process: after a cudaDeviceReset of that device (which tears down the
 * context the address belongs to) do not call this entry point there again.
 * The steps, launch counting and profiling records are moe_route's own: the
 * same router path (tensor cores for bf16 and MXFP8 layers, CUDA cores for
 * fp32) and the same split-K order, so every output equals moe_route's. Every call on a device shares the one
 * array and it keeps the last call's contents (each call writes every entry
 * it reads, so none needs clearing); calls whose GPU work overlaps (other
 * streams, other handles) race and must be serialised by the caller. The
 * handle's device must be current. Calls no CUDA allocation routine. */
moe_status moe_route_noalloc(moe_handle h, const void* x, int T, float* logits, int32_t* idx, float* gate,
                             int32_t* cnt, int32_t* off, int32_t* perm, int32_t* inv, void* stream);

/* Self-test of the device-side failure path (the pages describe no such call):
 * launches one block that waits, with the bounded wait every tcgen05 pipeline
 * of the library uses, on an mbarrier that nothing arrives at. After limit_ms
 * (1..10000) the wait gives up, MOE_ERR_TIMEOUT is recorded in the status word
 * (read it with moe_get_status) and the kernel returns; the CUDA context stays
 * usable. Asynchronous on `stream`. */
moe_status moe_selftest_timeout(moe_handle h, int limit_ms, void* stream);

/* Tracing. When enabled, every kernel launch of later calls on this handle is
 * bracketed by two CUDA events recorded on the call's stream (no extra device
 * memory). moe_profile_read waits for the recorded events and returns, for
 * each kernel group that ran (at most max_groups), its name (NUL-terminated,
 * at most 31 characters, in names[32*i]), its kernel launches and the summed
 * milliseconds between its events; then it forgets the records. *n_groups
 * receives the number of groups written. While enabled, every kernel runs on
 * the call's stream (no side-stream overlap in moe_backward), so that each
 * group's events bracket its own kernels. */
moe_status moe_profile_enable(moe_handle h, int enable);
moe_status moe_profile_read(moe_handle h, int max_groups, char* names, long long* launches, double* total_ms,
                            int* n_groups);

/* Number of kernels the handle has launched since moe_create (host counter). */
moe_status moe_launch_count(moe_handle h, long long* launches);

/* Human-readable name of a status code (static string). */
const char* moe_status_string(int status);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
