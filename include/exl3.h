/*
 * exl3.h -- C ABI of the GB300 (sm_103a) library for one routed-expert MoE
 * layer whose expert weights are EXL3 K-bit trellis codes.
 *
 * Sources (web pages, cited by title and section):
 *   [p1] "GLM-5.3-Flash EXL3 (~2.1 bpw, SM70 tile order)"
 *   [p2] "GLM-5.3 Flash EXL3 for 2x DGX Sparks"
 *   [p3] "GLM-5.3-Flash EXL3 K2"
 *   [p4] "GLM-5.3-Flash · exlr8 (K2/K3/K4)"
 *
 * Conventions for every entry point:
 *   - Tensors are caller-owned memory; "device" pointers must be CUDA device
 *     (or managed) memory of the current device, "host" pointers host memory.
 *     The library never frees them.  A layer handle borrows the weight
 *     pointers given to exl3_layer_create and must not outlive them.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Work is enqueued asynchronously; nothing synchronises the host
 *     unless stated.  exl3_moe_route and exl3_moe_forward never allocate and
 *     never read device data on the host, so they can be captured in a CUDA
 *     graph (the pages capture decode steps in graphs: [p2] What runs, Graphs).
 *   - Errors: argument, shape and width errors are returned before any launch
 *     and leave outputs untouched.  A failed launch returns EXL3_ERR_CUDA.
 *     Inconsistencies found on the device (bad expert id in a table, a wait
 *     that timed out) set a status word in the workspace, read back with
 *     exl3_get_device_status.
 *   - Layouts are row-major and densely packed unless stated.
 *
 * Format v1 (the library's reading of the pages, which name the format but
 * do not define its bits): codes of one projection of one expert are uint16 [in/16][out/16][16*K]
 * ([p1] intro: packed int16 words holding 16/K weights; [p4] Loading: 16x16
 * tiles, a 4096x128 half at width K is 65,536*K bytes); suh is fp16 [in],
 * svh fp16 [out] ([p2] What runs: trellis + suh + svh + mcg).
 */
#ifndef EXL3_H
#define EXL3_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct exl3_layer exl3_layer_t; /* opaque, immutable after create */

typedef enum {
    EXL3_OK = 0,
    EXL3_ERR_ARG = 1,       /* null pointer, bad enum, top_k out of range */
    EXL3_ERR_SHAPE = 2,     /* dimensions not multiples of 128, T < 0, ... */
    EXL3_ERR_K = 3,         /* code width not in {2, 3, 4} */
    EXL3_ERR_WORKSPACE = 4, /* workspace null or smaller than required */
    EXL3_ERR_CUDA = 5,      /* a CUDA call or launch failed */
    EXL3_ERR_DEVICE = 6     /* no sm_100-family device / device status set */
} exl3_status;

typedef enum { EXL3_F16 = 0, EXL3_BF16 = 1 } exl3_dtype;

/* Kernel path for the expert GEMMs.  AUTO picks the grouped GEMV for
 * decode-sized steps (few tokens per expert) and the tcgen05 grouped GEMM
 * for prefill-sized steps. */
typedef enum { EXL3_PATH_AUTO = 0, EXL3_PATH_GEMV = 1, EXL3_PATH_GEMM = 2 } exl3_path;

/* Projection index: 0 = gate, 1 = up, 2 = down. */
typedef struct {
    int num_experts;             /* E, 1..1024 */
    int hidden;                  /* H, multiple of 128 */
    int inter;                   /* I, multiple of 128 */
    int K[3];                    /* code width per projection, 2..4 */
    int fp8_round;               /* 1 = round codebook outputs to FP8 E4M3 before the side
                                    vectors ([p4] intro, the exlr8 rule) */
    uint32_t mcg_mult;           /* mcg multiplier (odd); 0 = 0x9E3779B1 */
    const uint16_t *codes[3];    /* device, [E][in/16][out/16][16*K[p]] */
    const uint16_t *suh[3];      /* device fp16 bits, [E][in] */
    const uint16_t *svh[3];      /* device fp16 bits, [E][out] */
    const uint16_t *shared_w[3]; /* device fp16 bits, dense [in][out], or all NULL: one
                                    unquantized shared expert added with weight 1
                                    ([p4] intro: one shared expert per MoE layer) */
    int hadamard;                /* 0 = format v1; 1 = format v2: the routed projections
                                    carry the 128-point Hadamard rotation on both sides,
                                    W_eff = diag(suh) Hb V Hb diag(svh), Hb block diagonal
                                    with copies of the normalized 128x128 Sylvester matrix,
                                    entries (-1)^popcount(i & j) / sqrt(128) ([p4]
                                    Calibration names the 128x128 Hadamard matrix as a
                                    format primitive).  Other values: EXL3_ERR_ARG */
    int shared_coded;            /* 1: the code, suh and svh arrays hold num_experts + 1
                                    experts, the last one a trellis-coded shared expert
                                    that every token uses with weight 1, after its routed
                                    pairs ([p4] Loading: the shared expert is stored as
                                    expert 288, after the routed experts, at their width).
                                    Requires shared_w all NULL and num_experts + 1 <= 1024.
                                    num_experts stays the router's width (logit columns). */
    const uint8_t *expert_K;     /* host, optional: [num_experts + shared_coded][3] code width
                                    (2..4) of every expert and projection ([p4] Loading: the
                                    bit201 and bit349 manifests give some experts or
                                    projections another width; [p5] Rates: every routed
                                    tensor K3 or K4).  With it K[] is ignored and codes[p]
                                    holds the experts' codes back to back: expert e at word
                                    offset sum over f < e of (in/16)(out/16)*16*expert_K[f][p].
                                    Copied at create (which then allocates two small device
                                    tables, freed by exl3_layer_destroy).  NULL: K[p] for
                                    every expert. */
    int act_fp8;                 /* 1: FP8 x FP8 products.  The activation operand of
                                    every routed projection (x * suh for gate and up,
                                    h * suh for down, after the rotation in format v2) is
                                    quantised per row to E4M3: s = amax / 448 and
                                    q = E4M3_RNE_sat(a / s), both divisions in IEEE fp32,
                                    and the product is s * sum q * v; the tensor-core
                                    path then multiplies E4M3 by E4M3 (tcgen05
                                    kind::f8f6f4).  Requires fp8_round = 1 (the weight
                                    operand is the E4M3 codebook value) ([p4] Widths: with
                                    the E4M3 codebook the prefill runs on FP8 tensor
                                    cores; the pages give no activation recipe, this is
                                    the library's reading).  The dense shared expert is
                                    not affected.  0: fp16 operands.  Other values, or 1
                                    without fp8_round: EXL3_ERR_ARG. */
} exl3_layer_desc;

/* Validate `desc` and build a handle.  codes, suh, svh and shared_w must be
 * 16-byte aligned.  Gate and up may differ in width (K[0] != K[1]): such a
 * layer, like one with expert_K, runs its expert kernels once per width over
 * device-built work lists.  A layer with a dense shared expert also
 * creates one CUDA stream and two events on the current device (released by
 * exl3_layer_destroy); the shared expert of every forward runs on that stream,
 * forked from the caller's stream after routing and joined before the
 * combine, so forwards on one handle must be issued by one host thread at a
 * time.  Errors:
 * EXL3_ERR_ARG (null pointers, shared_w partly NULL), EXL3_ERR_SHAPE,
 * EXL3_ERR_K, EXL3_ERR_DEVICE (current device is not compute capability
 * 10.x), EXL3_ERR_CUDA (stream or event creation failed). */
exl3_status exl3_layer_create(const exl3_layer_desc *desc, exl3_layer_t **out);
void exl3_layer_destroy(exl3_layer_t *layer);

/* Decode projection `proj` of `expert` (0 .. num_experts - 1 + shared_coded)
 * to a dense fp16 matrix out[in][out] (device).  apply_side = 0: the codebook values (after the E4M3 rule when the
 * layer has fp8_round); apply_side = 1: fp16(fp32(fp32(v*suh[i])*svh[o])).
 * The Hadamard rotation of format v2 is never applied here: this is the
 * element-wise, bit-exact check path for the codes ([p2] Cold prefill: the
 * dense "LinearEXL3 reference").  Errors: EXL3_ERR_ARG for bad expert/proj/null. */
exl3_status exl3_decode_dense(const exl3_layer_t *layer, int expert, int proj, int apply_side,
                              uint16_t *out, void *stream);

/* Bytes of workspace exl3_moe_route needs for T tokens, E experts, top_k. */
size_t exl3_route_workspace_size(int T, int E, int top_k);

/* Top-k routing and segment tables ([p4] intro: 288 experts, top-8; [p2] Cold
 * prefill (E3): device-side segment tables, no host sync).
 *   logits      device fp32 [T][E]
 *   ids         device int32 [T][top_k]  experts by descending logit, ties to
 *               the lower index, NaN as -inf
 *   w           device fp32 [T][top_k]   softmax over the k selected logits
 *   seg_offsets device int32 [E+1]       pairs with expert < e
 *   seg_pairs   device int32 [T*top_k]   pair ids t*top_k+j, expert-major,
 *               ascending inside an expert
 *   ws          device, >= exl3_route_workspace_size bytes
 * T = 0 is valid (offsets all zero).  1 <= top_k <= min(E, 16). */
exl3_status exl3_moe_route(const float *logits, int T, int E, int top_k, int32_t *ids, float *w,
                           int32_t *seg_offsets, int32_t *seg_pairs, void *ws, size_t ws_bytes,
                           void *stream);

/* Size of the device array behind exl3_moe_route_static: 1 MiB, held on every
 * device that loads this library until the process exits. */
#define EXL3_ROUTE_STATIC_SCRATCH_BYTES (1u << 20)

/* exl3_moe_route without a workspace argument.  The pages have no counterpart:
 * it exists for callers that cannot allocate device memory themselves, such
 * as a plugin whose host framework owns every device allocation and hands out
 * only the tensors of the call, or a loop that must not call cudaMalloc
 * because cudaMalloc can synchronise the device.  The caller still provides
 * logits and the four outputs, with the layouts, rules and errors of
 * exl3_moe_route; the routing scratch is instead a library-owned device array
 * of EXL3_ROUTE_STATIC_SCRATCH_BYTES.  No call allocates or frees memory.
 *   - Sizes whose exl3_route_workspace_size(T, E, top_k) exceeds
 *     EXL3_ROUTE_STATIC_SCRATCH_BYTES return EXL3_ERR_SHAPE before any launch;
 *     any T <= 4096 with E <= 1024 and top_k <= 16 fits.
 *   - The first call on a device looks up the array's device address
 *     (once per device, with that device current); make that first call
 *     before any stream capture begins.  The address is kept for the life
 *     of the process, so every call must run in the device's primary
 *     context (the CUDA runtime's default): not after cudaDeviceReset, and
 *     not under a context the caller created and made current.
 *   - Every call on a device shares the one array, and it keeps the last
 *     call's contents.  Each call clears what has to start at zero, but calls
 *     whose work overlaps on the GPU (different streams without ordering,
 *     several host threads) race on it: order them on one stream.
 *   - The device status word lives in that array, so exl3_get_device_status
 *     cannot read it. */
exl3_status exl3_moe_route_static(const float *logits, int T, int E, int top_k, int32_t *ids,
                                  float *w, int32_t *seg_offsets, int32_t *seg_pairs,
                                  void *stream);

/* Bytes of workspace exl3_moe_forward needs for T tokens and top_k (all
 * paths).  Deterministic in (layer shape, T, top_k). */
size_t exl3_moe_workspace_size(const exl3_layer_t *layer, int T, int top_k);

/* One MoE layer forward ([p2] Cold prefill (E3): gather, gate/up + SwiGLU,
 * down + scatter; [p1] Running it: decodes the trellis inside the matmul):
 *   x      device [T][H] in dtype dt (fp16 or bf16)
 *   logits device fp32 [T][E], E = num_experts (routed experts)
 *   out    device [T][H] in dtype dt; y_t = sum_j w_tj * expert_{id_tj}(x_t)
 *          (+ shared(x_t)), summed over j in order, no atomics; a coded
 *          shared expert is the last term, a dense one is added after it
 *   ws     device workspace of >= exl3_moe_workspace_size(layer, T, top_k)
 * out may not alias x. */
exl3_status exl3_moe_forward(const exl3_layer_t *layer, const void *x, exl3_dtype dt,
                             const float *logits, int T, int top_k, void *out, void *ws,
                             size_t ws_bytes, void *stream);

/* As exl3_moe_forward, plus an optional residual (device [T][H] in dt, may
 * be NULL; out = round(residual + y)) and an explicit kernel path.
 * Both return EXL3_ERR_SHAPE for T > 262,136 on a layer with a dense shared
 * expert (its launches cover 8 tokens per grid slice), and for more than 2^29
 * (token, expert) pairs (2^26 on the decode-sized GEMV path; exl3_moe_route
 * takes 2^29 too). */
exl3_status exl3_moe_forward_ex(const exl3_layer_t *layer, const void *x, exl3_dtype dt,
                                const float *logits, int T, int top_k, const void *residual,
                                void *out, int path, void *ws, size_t ws_bytes, void *stream);

/* One layer forward over a range of experts, for expert parallelism
 * (expert-parallel sharding of the routed experts over N ranks; the pages
 * split the layer over GPUs and sum the partial outputs with one
 * all-reduce per layer: [p2] Why the overlay exists).  Routing covers every
 * token and expert as in exl3_moe_forward; only the (token, expert) pairs
 * whose expert e has expert_begin <= e < expert_end are computed (with a
 * coded shared expert, its index is num_experts, the last one), plus the
 * dense shared expert when with_shared = 1.  out (device fp32 [T][H]) gets
 * their unrounded sum, summed in pair order, so the ranks' outputs summed
 * over a partition of [0, num_experts + shared_coded) with the shared expert
 * on exactly one rank give the layer before its final rounding (finish with
 * exl3_round_output).  The workspace and path are as for
 * exl3_moe_forward_ex.  Errors: those of exl3_moe_forward_ex, and
 * EXL3_ERR_ARG for a range outside [0, num_experts + shared_coded] or
 * with_shared not 0 / 1. */
exl3_status exl3_moe_forward_experts(const exl3_layer_t *layer, const void *x, exl3_dtype dt,
                                     const float *logits, int T, int top_k, int expert_begin,
                                     int expert_end, int with_shared, float *out, int path,
                                     void *ws, size_t ws_bytes, void *stream);

/* out = round(y + residual) to dt: the last step of a layer whose partial
 * sums were reduced outside the library.  y device fp32 [T][H], residual
 * device [T][H] in dt or NULL, out device [T][H] in dt; all 16-byte aligned,
 * H a multiple of 4. */
exl3_status exl3_round_output(const float *y, int T, int H, const void *residual, exl3_dtype dt,
                              void *out, void *stream);

/* Unweighted RMSNorm of each row: out = round(x / sqrt(mean(x^2) + eps)),
 * fp32 arithmetic, x and out device [T][H] in dt (out may alias x).  Used
 * between layers of a stacked prefill. */
exl3_status exl3_rmsnorm(const void *x, exl3_dtype dt, int T, int H, float eps, void *out,
                         void *stream);

/* Synchronise `stream` and read the device status word of a forward/route
 * workspace (0 = fine). */
exl3_status exl3_get_device_status(const void *ws, void *stream, int32_t *status);

/* Stage-boundary profiling.  When set, every forward on this layer records
 * events[i] (cudaEvent_t, created by the caller) on its stream at these
 * boundaries: 0 start, 1 routing done, 2 gather done, 3 gate/up done,
 * 4 down input prepared, 5 down done, 6 joined with the shared expert's
 * stream, 7 combine done.
 * n_events must be EXL3_NUM_STAGE_EVENTS; events = NULL clears the hook.
 * For measurement only: not safe while another thread runs a forward on the
 * same layer. */
#define EXL3_NUM_STAGE_EVENTS 8
exl3_status exl3_layer_set_stage_events(exl3_layer_t *layer, void *const *events, int n_events);

/* Number of kernels this library has launched in the process so far (a
 * host-side counter; launches captured into a CUDA graph count once, at
 * capture). */
uint64_t exl3_launch_count(void);

/* The per-row E4M3 quantisation of a layer with act_fp8 = 1, on its own:
 * for each of `rows` rows of `n` fp32 values a (device, row-major), the row
 * scale s = fp32(amax / 448) (0 for an all-zero row) and the E4M3 bytes
 * q_i = E4M3_RNE_sat(fp32(a_i / s)) (0 when s = 0), the decisions the
 * activation passes of the FP8 path take ([p4] Widths: FP8 tensor cores; the
 * recipe is the library's reading).  q: device uint8 [rows][n]; s: device
 * fp32 [rows].  Errors: EXL3_ERR_SHAPE for negative sizes, EXL3_ERR_ARG for
 * null pointers, EXL3_ERR_CUDA for a failed launch. */
exl3_status exl3_quantize_rows_e4m3(const float *a, int rows, int n, uint8_t *q, float *s,
                                    void *stream);

/* Test hook for the bounded waits of the tensor-core kernels (the pages have
 * no counterpart).  Every wait inside those kernels has a clock budget; when
 * one runs out, the kernel sets bit 4 (value 4) of the device status word,
 * every CTA of the grid stops issuing work, drains the copies and tensor-core
 * operations it already issued, frees its TMEM and returns, and
 * exl3_get_device_status then reports EXL3_ERR_DEVICE with that bit.  This
 * hook makes such a wait run out on purpose, without any fault: in the
 * gate/up launch of the chosen kernel (1 = big tiles of more than 128
 * tokens, 2 = small tiles of at most 128 tokens) the thread that loads the
 * activation operands skips K step `ks` (64 inputs per step; a step past the
 * end has no effect), so the MMA issuer waits on a barrier that nothing
 * completes, and every wait of that launch gets `budget_cycles` SM clock
 * cycles (100,000 .. 1,000,000,000) instead of the default 1,000,000,000.
 * kernel = 0 clears the hook.  It stays set for every later forward of the
 * process; a forward run with it gives an unspecified output.  Not thread
 * safe.  Errors: EXL3_ERR_ARG for values outside these ranges. */
exl3_status exl3_test_set_wait_fault(int kernel, int ks, long long budget_cycles);

const char *exl3_status_string(exl3_status s);

#ifdef __cplusplus
}
#endif

#endif /* EXL3_H */
