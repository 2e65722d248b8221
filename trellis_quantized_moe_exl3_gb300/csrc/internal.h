// Internal launch interface between the C ABI (layer.cu) and the kernels.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/exl3.h"

namespace exl3 {

// Host-side count of kernel launches (exl3_launch_count).
void note_launches(int n);

// Record a profiling event; inside stream capture it becomes an external
// event node, so it can still be timed after graph replay.
inline void record_stage_event(cudaEvent_t ev, cudaStream_t st) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaStreamIsCapturing(st, &cs);
  if (cs == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(ev, st, cudaEventRecordExternal);
  else
    cudaEventRecord(ev, st);
}

// Launch with programmatic dependent launch allowed (see pdl_wait).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

constexpr uint32_t kDefaultMcgMult = 0x9E3779B1u;
constexpr int kRouteChunk = 64;    // tokens per routing CTA
constexpr int kMaxTopK = 16;
constexpr int kMaxExperts = 1024;
constexpr int kGroup = 8;          // tokens per GEMV token group (MMA N)
// Pairs (tokens x top_k) a call may hold: positions and TMA row coordinates
// are 32-bit (the GEMM path addresses 2 x pairs rows); the GEMV path forms
// split x projection x pairs row indices, so it takes 32 times fewer.
constexpr size_t kMaxPairs = (size_t)1 << 29;
constexpr size_t kMaxGemvPairs = (size_t)1 << 26;

// Device status bits (workspace status word).
enum : int32_t {
  kStatusBadExpert = 1,   // an expert id outside [0, E) reached a kernel
  kStatusBadSegment = 2,  // a segment table entry out of range
  kStatusTimeout = 4,     // a bounded wait gave up
};

struct RouteBuffers {
  int32_t* ids;          // [P]
  float* w;              // [P]
  int32_t* seg_offsets;  // [E+1]
  int32_t* seg_pairs;    // [P]
  int32_t* pair_pos;     // [P]  position of pair p in seg_pairs
  int32_t* active;       // [E+1]: active[0] = count, active[1..] = experts with pairs
  int32_t* chunk_counts; // [nchunks][E]
  int32_t* rank;         // [P]
  int32_t* status;       // [1]
  int32_t* group_off;    // [E+1]: first token group of each expert; [E] = number of groups
  int32_t* groups;       // [max_groups][4]: {expert, first position, count, 0}
};

// Upper bound on the number of kGroup-token groups over all experts.
inline size_t max_groups(int T, int E, int top_k) {
  const size_t P = (size_t)T * top_k;
  const size_t a = (P + kGroup - 1) / kGroup + ((size_t)E < P ? (size_t)E : P);
  return a < P ? a : P;
}

// E and top_k here count every table entry: with a coded shared expert,
// E + 1 experts and top_k + 1 pairs per token.
size_t route_scratch_bytes(int T, int E, int top_k);
// Carves RouteBuffers out of `ws` (ids/w/seg may be caller-provided: non-null
// fields of `given` are kept).
void route_carve(void* ws, int T, int E, int top_k, RouteBuffers* rb);
// E = logits per token, top_k = routed pairs per token; shared = 1 appends
// pair (expert E, weight 1) to every token (tables of E + 1 experts,
// top_k + 1 pairs per token).
cudaError_t launch_route(const float* logits, int T, int E, int top_k, const RouteBuffers& rb,
                         cudaStream_t st, int shared = 0);

// Expert range of one call: only (token, expert) pairs whose expert e has
// e0 <= e < e1 are computed and summed (expert parallelism: each rank takes
// a range, the ranks' partial outputs are summed).  [0, E) is the whole layer.
struct Shard {
  int e0, e1;
};

struct LayerView {
  int E, H, I;
  int K[3];
  int fp8;
  uint32_t mult;
  const uint16_t* codes[3];
  const uint16_t* suh[3];
  const uint16_t* svh[3];
  const uint16_t* shared_w[3];
  size_t code_stride[3];  // uint16 words per expert
  int had;                // format v2: Hadamard rotation on both sides of each projection
  int act8;               // FP8 operand mode: every projection's activation row is
                          // quantised to E4M3 with an fp32 row scale (requires fp8)
  int sc;                 // 1: expert E - 1 of the arrays is the coded shared expert
                          // (E counts it; the logits have E - sc columns)
  // Mixed widths (a width per expert and projection, or gate and up of
  // different widths): the expert kernels run once per width over work lists.
  int mixed;
  const int32_t* d_kt;             // device [E][3] widths
  const unsigned long long* d_off; // device [E][3] code word offsets
  const uint8_t* h_kt;             // host copies of both
  const size_t* h_off;
  int wmask[2];                    // widths present (bit K - 2): [0] gate/up, [1] down
};

// Width of projection p of expert e and the word offset of its codes.
inline int layer_width(const LayerView& L, int e, int p) {
  return L.mixed ? L.h_kt[(size_t)e * 3 + p] : L.K[p];
}
inline size_t layer_code_offset(const LayerView& L, int e, int p) {
  return L.mixed ? L.h_off[(size_t)e * 3 + p] : L.code_stride[p] * (size_t)e;
}

cudaError_t launch_decode_dense(const LayerView& L, int expert, int proj, int apply_side,
                                uint16_t* out, cudaStream_t st);

// ---- grouped GEMV path (decode-sized steps)
struct GemvBuffers {
  uint32_t* xs_gu;   // [group][2][H/16][8][16] fp16x2 (dup), permuted per 16-block
  float* xs_gu_inv;  // [P][2]
  float* gu;         // [ns_gu][2][P][I] fp32 gate and up K-split partials (pair-sorted rows)
  uint32_t* xs_d;    // [group][I/16][8][16] fp16x2 (dup), permuted
  float* xs_d_inv;   // [P]
  float* r;          // [ns_d][P][H] fp32 K-split partial rows by pair id
  int32_t* counters; // item counters: [launch (gate/up, down)][width 2..4]
  int32_t* n_entries;  // mixed widths: entries per [launch][width]
  int32_t* entries;    // mixed widths: (group, projection) pairs, [launch][width][cap]
  int ns_gu, ns_d;   // K splits of the two launches
};
size_t gemv_scratch_bytes(int T, int top_k, int E, int H, int I);
void gemv_carve(void* ws, int T, int top_k, int E, int H, int I, GemvBuffers* gb);
// ev (may be null): events recorded after gather [2], gate/up [3], down prep [4], down [5].
cudaError_t launch_moe_gemv(const LayerView& L, const void* x, int x_bf16, int T, int top_k,
                            const RouteBuffers& rb, const GemvBuffers& gb, const cudaEvent_t* ev,
                            Shard sh, cudaStream_t st);

// ---- grouped GEMM path (prefill-sized steps, tcgen05)
size_t gemm_scratch_bytes(int T, int top_k, int E, int H, int I, int had, int act8);
// ev (may be null): events after gather [2], gate/up [3], down input [4], down [5].
// *r_out receives the pair-row buffer [P][H] the combine reads.
cudaError_t launch_moe_gemm(const LayerView& L, const void* x, int x_bf16, int T, int top_k,
                            const RouteBuffers& rb, void* ws, const cudaEvent_t* ev, float** r_out,
                            Shard sh, cudaStream_t st);

// ---- shared expert (dense fp16)
size_t shared_scratch_bytes(int T, int H, int I);
// scratch: shared_scratch_bytes(T, H, I) bytes.  *part_d / *nsplit_d receive
// the down projection's partial sums [nsplit][T][H] that the combine adds.
cudaError_t launch_shared(const LayerView& L, const void* x, int x_bf16, int T, void* scratch,
                          const float** part_d, int* nsplit_d, cudaStream_t st);

// ---- combine / norm
// r: [r_splits][T*top_k][H] pair rows (K-split partials, added in order);
// only pairs whose expert (ids) lies in the shard's range are added.
// out_f32: out is fp32 and takes the sum unrounded (no residual).
cudaError_t launch_combine(const float* r, int r_splits, int T, int top_k, int H,
                           const int32_t* ids, Shard sh, const float* shared_part,
                           int shared_splits, const void* residual, void* out, int out_bf16,
                           int out_f32, cudaStream_t st);
// out = round(y + residual) to bf16 / fp16 (y fp32 [T][H]; residual may be null).
cudaError_t launch_round_output(const float* y, int T, int H, const void* residual, void* out,
                                int out_bf16, cudaStream_t st);
cudaError_t launch_rmsnorm(const void* x, int bf16, int T, int H, float eps, void* out,
                           cudaStream_t st);

}  // namespace exl3
