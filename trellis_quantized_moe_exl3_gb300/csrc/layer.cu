// C ABI of the EXL3 MoE library: argument validation, workspace layout and
// the launch sequence of one layer forward.  See include/exl3.h for the
// contract of each entry point.
#include <stdlib.h>
#include <string.h>

#include <atomic>

#include "internal.h"

using namespace exl3;

struct exl3_layer {
  LayerView v;
  int has_shared;
  cudaEvent_t ev[EXL3_NUM_STAGE_EVENTS];
  int has_ev;
  // the shared expert runs on a side stream, forked from and joined to the
  // caller's stream inside each forward
  cudaStream_t side;
  cudaEvent_t fork, join;
  // mixed widths: owned width / offset tables (host and device copies)
  uint8_t* h_kt;
  size_t* h_off;
  int32_t* d_kt;
  unsigned long long* d_off;
};

namespace {
std::atomic<uint64_t> g_launches{0};
}

void exl3::note_launches(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

namespace {

size_t al(size_t b) { return (b + 255) & ~(size_t)255; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

exl3_status check_device() {
  int dev = 0, major = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return EXL3_ERR_DEVICE;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess)
    return EXL3_ERR_DEVICE;
  return major == 10 ? EXL3_OK : EXL3_ERR_DEVICE;
}

// Forward workspace: [route scratch][ids][w][seg_offsets][seg_pairs][expert path][shared]
// The expert-path region holds the larger of the GEMV and GEMM scratch.
struct FwdLayout {
  size_t route, ids, w, off, pairs, gemv, shared, total;
};

// AUTO path: the tensor-core GEMM once an expert sees ~16 tokens on average.
bool use_gemm(const LayerView& L, int T, int top_k, int path) {
  if (path == EXL3_PATH_GEMV) return false;
  if (path == EXL3_PATH_GEMM) return true;
  return (size_t)T * top_k >= (size_t)16 * L.E;
}

// k = routed pairs per token; the tables hold k + L.sc (the coded shared
// expert's pair) per token over L.E experts.
FwdLayout fwd_layout(const LayerView& L, int has_shared, int T, int k_routed) {
  FwdLayout f{};
  const int k = k_routed + L.sc;
  const size_t P = (size_t)T * k;
  size_t o = 0;
  f.route = o; o += al(route_scratch_bytes(T, L.E, k));
  f.ids = o; o += al(P * 4);
  f.w = o; o += al(P * 4);
  f.off = o; o += al((size_t)(L.E + 1) * 4);
  f.pairs = o; o += al(P * 4);
  const size_t gv = gemv_scratch_bytes(T, k, L.E, L.H, L.I);
  const size_t gm = gemm_scratch_bytes(T, k, L.E, L.H, L.I, L.had, L.act8);
  f.gemv = o; o += al(gv > gm ? gv : gm);
  f.shared = o; o += has_shared ? al(shared_scratch_bytes(T, L.H, L.I)) : 0;
  f.total = o;
  return f;
}

}  // namespace

extern "C" {

const char* exl3_status_string(exl3_status s) {
  switch (s) {
    case EXL3_OK: return "ok";
    case EXL3_ERR_ARG: return "invalid argument";
    case EXL3_ERR_SHAPE: return "invalid shape";
    case EXL3_ERR_K: return "code width must be 2, 3 or 4";
    case EXL3_ERR_WORKSPACE: return "workspace missing or too small";
    case EXL3_ERR_CUDA: return "CUDA error";
    case EXL3_ERR_DEVICE: return "unsupported device or device status set";
  }
  return "unknown status";
}

exl3_status exl3_layer_create(const exl3_layer_desc* d, exl3_layer_t** out) {
  if (!d || !out) return EXL3_ERR_ARG;
  *out = nullptr;
  if (d->num_experts < 1 || d->num_experts > kMaxExperts) return EXL3_ERR_SHAPE;
  if (d->hidden <= 0 || d->inter <= 0 || d->hidden % 128 || d->inter % 128) return EXL3_ERR_SHAPE;
  if (d->shared_coded != 0 && d->shared_coded != 1) return EXL3_ERR_ARG;
  const int n_coded = d->num_experts + d->shared_coded;  // experts in the arrays
  if (d->expert_K) {
    for (int i = 0; i < 3 * n_coded; i++)
      if (d->expert_K[i] < 2 || d->expert_K[i] > 4) return EXL3_ERR_K;
  } else {
    for (int p = 0; p < 3; p++)
      if (d->K[p] < 2 || d->K[p] > 4) return EXL3_ERR_K;
  }
  const uint32_t mult = d->mcg_mult ? d->mcg_mult : kDefaultMcgMult;
  if (!(mult & 1u)) return EXL3_ERR_ARG;
  int nshared = 0;
  if (d->hadamard != 0 && d->hadamard != 1) return EXL3_ERR_ARG;
  if (d->act_fp8 != 0 && d->act_fp8 != 1) return EXL3_ERR_ARG;
  if (d->act_fp8 && !d->fp8_round) return EXL3_ERR_ARG;
  if (n_coded > kMaxExperts) return EXL3_ERR_SHAPE;
  for (int p = 0; p < 3; p++) {
    if (!d->codes[p] || !d->suh[p] || !d->svh[p]) return EXL3_ERR_ARG;
    if (!aligned16(d->codes[p]) || !aligned16(d->suh[p]) || !aligned16(d->svh[p]))
      return EXL3_ERR_ARG;
    nshared += d->shared_w[p] != nullptr;
    if (d->shared_w[p] && !aligned16(d->shared_w[p])) return EXL3_ERR_ARG;
  }
  if (nshared != 0 && nshared != 3) return EXL3_ERR_ARG;
  if (nshared && d->shared_coded) return EXL3_ERR_ARG;  // one shared expert at most
  exl3_status ds = check_device();
  if (ds != EXL3_OK) return ds;
  exl3_layer* L = static_cast<exl3_layer*>(calloc(1, sizeof(exl3_layer)));
  if (!L) return EXL3_ERR_ARG;
  LayerView& v = L->v;
  v.sc = d->shared_coded;
  v.E = d->num_experts + v.sc; v.H = d->hidden; v.I = d->inter;
  v.fp8 = d->fp8_round ? 1 : 0;
  v.mult = mult;
  v.had = d->hadamard;
  v.act8 = d->act_fp8;
  for (int p = 0; p < 3; p++) {
    v.K[p] = d->expert_K ? d->expert_K[p] : d->K[p];
    v.codes[p] = d->codes[p];
    v.suh[p] = d->suh[p];
    v.svh[p] = d->svh[p];
    v.shared_w[p] = d->shared_w[p];
    const size_t in = p == 2 ? v.I : v.H, outf = p == 2 ? v.H : v.I;
    v.code_stride[p] = (in / 16) * (outf / 16) * 16 * (size_t)v.K[p];
  }
  // Mixed widths: a width per expert and projection (expert_K), or gate and
  // up of different widths.  Codes of a projection lie expert after expert,
  // each at its own width, so the offsets are running sums.
  v.mixed = d->expert_K != nullptr || d->K[0] != d->K[1];
  if (v.mixed) {
    const size_t n = (size_t)3 * n_coded;
    L->h_kt = static_cast<uint8_t*>(malloc(n));
    L->h_off = static_cast<size_t*>(malloc(n * sizeof(size_t)));
    int32_t* kt32 = static_cast<int32_t*>(malloc(n * sizeof(int32_t)));
    unsigned long long* off64 = static_cast<unsigned long long*>(malloc(n * sizeof(unsigned long long)));
    bool ok = L->h_kt && L->h_off && kt32 && off64;
    if (ok) {
      size_t run[3] = {0, 0, 0};
      for (int e = 0; e < n_coded; e++)
        for (int p = 0; p < 3; p++) {
          const int k = d->expert_K ? d->expert_K[(size_t)e * 3 + p] : d->K[p];
          const size_t in = p == 2 ? v.I : v.H, outf = p == 2 ? v.H : v.I;
          L->h_kt[(size_t)e * 3 + p] = (uint8_t)k;
          v.wmask[p == 2 ? 1 : 0] |= 1 << (k - 2);
          kt32[(size_t)e * 3 + p] = k;
          L->h_off[(size_t)e * 3 + p] = run[p];
          off64[(size_t)e * 3 + p] = run[p];
          run[p] += (in / 16) * (outf / 16) * 16 * (size_t)k;
        }
      ok = cudaMalloc(&L->d_kt, n * sizeof(int32_t)) == cudaSuccess &&
           cudaMalloc(&L->d_off, n * sizeof(unsigned long long)) == cudaSuccess &&
           cudaMemcpy(L->d_kt, kt32, n * sizeof(int32_t), cudaMemcpyHostToDevice) == cudaSuccess &&
           cudaMemcpy(L->d_off, off64, n * sizeof(unsigned long long), cudaMemcpyHostToDevice) ==
               cudaSuccess;
    }
    free(kt32);
    free(off64);
    v.h_kt = L->h_kt;
    v.h_off = L->h_off;
    v.d_kt = L->d_kt;
    v.d_off = L->d_off;
    if (!ok) {
      exl3_layer_destroy(L);
      return EXL3_ERR_CUDA;
    }
  }
  L->has_shared = nshared == 3;
  if (L->has_shared) {
    if (cudaStreamCreateWithFlags(&L->side, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&L->fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&L->join, cudaEventDisableTiming) != cudaSuccess) {
      exl3_layer_destroy(L);
      return EXL3_ERR_CUDA;
    }
  }
  *out = L;
  return EXL3_OK;
}

void exl3_layer_destroy(exl3_layer_t* layer) {
  if (!layer) return;
  if (layer->side) cudaStreamDestroy(layer->side);
  if (layer->fork) cudaEventDestroy(layer->fork);
  if (layer->join) cudaEventDestroy(layer->join);
  if (layer->d_kt) cudaFree(layer->d_kt);
  if (layer->d_off) cudaFree(layer->d_off);
  free(layer->h_kt);
  free(layer->h_off);
  free(layer);
}

exl3_status exl3_decode_dense(const exl3_layer_t* layer, int expert, int proj, int apply_side,
                              uint16_t* out, void* stream) {
  if (!layer || !out || proj < 0 || proj > 2 || expert < 0 || expert >= layer->v.E)
    return EXL3_ERR_ARG;
  if (launch_decode_dense(layer->v, expert, proj, apply_side ? 1 : 0, out,
                          static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return EXL3_ERR_CUDA;
  return EXL3_OK;
}

size_t exl3_route_workspace_size(int T, int E, int top_k) {
  if (T < 0 || E < 1 || top_k < 1) return 0;
  return route_scratch_bytes(T, E, top_k);
}

exl3_status exl3_moe_route(const float* logits, int T, int E, int top_k, int32_t* ids, float* w,
                           int32_t* seg_offsets, int32_t* seg_pairs, void* ws, size_t ws_bytes,
                           void* stream) {
  if (T < 0 || E < 1 || E > kMaxExperts) return EXL3_ERR_SHAPE;
  if (top_k < 1 || top_k > kMaxTopK || top_k > E) return EXL3_ERR_ARG;
  if ((size_t)T * (size_t)top_k > kMaxPairs) return EXL3_ERR_SHAPE;
  if (!seg_offsets || !ws) return ws ? EXL3_ERR_ARG : EXL3_ERR_WORKSPACE;
  if (T > 0 && (!logits || !ids || !w || !seg_pairs)) return EXL3_ERR_ARG;
  if (ws_bytes < route_scratch_bytes(T, E, top_k)) return EXL3_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  RouteBuffers rb{};
  route_carve(ws, T, E, top_k, &rb);
  rb.ids = ids; rb.w = w; rb.seg_offsets = seg_offsets; rb.seg_pairs = seg_pairs;
  if (launch_route(logits, T, E, top_k, rb, st) != cudaSuccess) return EXL3_ERR_CUDA;
  return EXL3_OK;
}

size_t exl3_moe_workspace_size(const exl3_layer_t* layer, int T, int top_k) {
  if (!layer || T < 0 || top_k < 1) return 0;
  return fwd_layout(layer->v, layer->has_shared, T, top_k).total;
}

}  // extern "C"

namespace {

// One forward over the experts of `sh` (all of them for a whole layer).
// with_shared: add the dense shared expert; out_f32: out is the fp32 sum
// (no residual, no rounding), else round(residual + sum) in dt.
exl3_status forward_impl(const exl3_layer_t* layer, const void* x, exl3_dtype dt,
                         const float* logits, int T, int top_k, const void* residual, void* out,
                         int path, void* ws, size_t ws_bytes, void* stream, Shard sh,
                         int with_shared, int out_f32) {
  if (!layer) return EXL3_ERR_ARG;
  const LayerView& L = layer->v;
  if (dt != EXL3_F16 && dt != EXL3_BF16) return EXL3_ERR_ARG;
  if (path < EXL3_PATH_AUTO || path > EXL3_PATH_GEMM) return EXL3_ERR_ARG;
  if (T < 0) return EXL3_ERR_SHAPE;
  if (top_k < 1 || top_k > kMaxTopK || top_k > L.E - L.sc) return EXL3_ERR_ARG;
  const size_t pairs = (size_t)T * (size_t)(top_k + L.sc);
  if (pairs > kMaxPairs || (!use_gemm(L, T, top_k + L.sc, path) && pairs > kMaxGemvPairs))
    return EXL3_ERR_SHAPE;
  if (T == 0) return EXL3_OK;
  if (!x || !logits || !out) return EXL3_ERR_ARG;
  if (!aligned16(x) || !aligned16(out) || (residual && !aligned16(residual))) return EXL3_ERR_ARG;
  if (x == out) return EXL3_ERR_ARG;
  const bool run_shared = layer->has_shared && with_shared;
  // the dense shared expert's gate/up launch has a grid z of 2 * ceil(T / 8)
  if (layer->has_shared && (size_t)T > (size_t)8 * (65535 / 2)) return EXL3_ERR_SHAPE;
  const FwdLayout f = fwd_layout(L, layer->has_shared, T, top_k);
  if (!ws) return EXL3_ERR_WORKSPACE;
  if (ws_bytes < f.total) return EXL3_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* base = static_cast<char*>(ws);
  // with a coded shared expert every token has one more pair (expert E - 1,
  // weight 1), and from here on the expert kernels see kp pairs per token
  const int kp = top_k + L.sc;
  RouteBuffers rb{};
  route_carve(base + f.route, T, L.E, kp, &rb);
  rb.ids = reinterpret_cast<int32_t*>(base + f.ids);
  rb.w = reinterpret_cast<float*>(base + f.w);
  rb.seg_offsets = reinterpret_cast<int32_t*>(base + f.off);
  rb.seg_pairs = reinterpret_cast<int32_t*>(base + f.pairs);
  const int bf16 = dt == EXL3_BF16;

  const cudaEvent_t* ev = layer->has_ev ? layer->ev : nullptr;
  auto rec = [&](int i) {
    if (ev) record_stage_event(ev[i], st);
  };
  // shared expert: on the side stream, joined before the combine.  With the
  // GEMV path it is forked before routing: the GEMV launches are persistent
  // grids that take the SMs as the kernel before them ends and keep them
  // until their work list is empty, so a kernel forked after routing would
  // mostly wait for them.  With the GEMM path it is forked once routing is
  // done, so it does not delay the routing CTAs.
  const bool gemm = use_gemm(L, T, kp, path);
  const float* sp = nullptr;
  int ns = 0;
  auto fork_shared = [&]() -> bool {
    return cudaEventRecord(layer->fork, st) == cudaSuccess &&
           cudaStreamWaitEvent(layer->side, layer->fork, 0) == cudaSuccess &&
           launch_shared(L, x, bf16, T, base + f.shared, &sp, &ns, layer->side) == cudaSuccess &&
           cudaEventRecord(layer->join, layer->side) == cudaSuccess;
  };
  rec(0);
  if (run_shared && !gemm && !fork_shared()) return EXL3_ERR_CUDA;
  if (launch_route(logits, T, L.E - L.sc, top_k, rb, st, L.sc) != cudaSuccess)
    return EXL3_ERR_CUDA;
  if (run_shared && gemm && !fork_shared()) return EXL3_ERR_CUDA;
  rec(1);

  float* pair_rows = nullptr;
  int pair_splits = 1;
  if (gemm) {
    if (launch_moe_gemm(L, x, bf16, T, kp, rb, base + f.gemv, ev, &pair_rows, sh, st) !=
        cudaSuccess)
      return EXL3_ERR_CUDA;
  } else {
    GemvBuffers gb{};
    gemv_carve(base + f.gemv, T, kp, L.E, L.H, L.I, &gb);
    if (launch_moe_gemv(L, x, bf16, T, kp, rb, gb, ev, sh, st) != cudaSuccess) return EXL3_ERR_CUDA;
    pair_rows = gb.r;
    pair_splits = gb.ns_d;
  }

  if (run_shared && cudaStreamWaitEvent(st, layer->join, 0) != cudaSuccess)
    return EXL3_ERR_CUDA;
  rec(6);
  if (launch_combine(pair_rows, pair_splits, T, kp, L.H, rb.ids, sh, sp, ns,
                     out_f32 ? nullptr : residual, out, bf16, out_f32, st) != cudaSuccess)
    return EXL3_ERR_CUDA;
  rec(7);
  return EXL3_OK;
}

}  // namespace

extern "C" {

exl3_status exl3_moe_forward_ex(const exl3_layer_t* layer, const void* x, exl3_dtype dt,
                                const float* logits, int T, int top_k, const void* residual,
                                void* out, int path, void* ws, size_t ws_bytes, void* stream) {
  if (!layer) return EXL3_ERR_ARG;
  return forward_impl(layer, x, dt, logits, T, top_k, residual, out, path, ws, ws_bytes, stream,
                      Shard{0, layer->v.E}, 1, 0);
}

exl3_status exl3_moe_forward_experts(const exl3_layer_t* layer, const void* x, exl3_dtype dt,
                                     const float* logits, int T, int top_k, int expert_begin,
                                     int expert_end, int with_shared, float* out, int path,
                                     void* ws, size_t ws_bytes, void* stream) {
  if (!layer) return EXL3_ERR_ARG;
  if (expert_begin < 0 || expert_end > layer->v.E || expert_begin > expert_end)
    return EXL3_ERR_ARG;
  if (with_shared != 0 && with_shared != 1) return EXL3_ERR_ARG;
  return forward_impl(layer, x, dt, logits, T, top_k, nullptr, out, path, ws, ws_bytes, stream,
                      Shard{expert_begin, expert_end}, with_shared, 1);
}

exl3_status exl3_round_output(const float* y, int T, int H, const void* residual, exl3_dtype dt,
                              void* out, void* stream) {
  if (dt != EXL3_F16 && dt != EXL3_BF16) return EXL3_ERR_ARG;
  if (T < 0 || H <= 0 || H % 4) return EXL3_ERR_SHAPE;
  if (T == 0) return EXL3_OK;
  if (!y || !out || !aligned16(y) || !aligned16(out) || (residual && !aligned16(residual)))
    return EXL3_ERR_ARG;
  if (launch_round_output(y, T, H, residual, out, dt == EXL3_BF16,
                          static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return EXL3_ERR_CUDA;
  return EXL3_OK;
}

exl3_status exl3_moe_forward(const exl3_layer_t* layer, const void* x, exl3_dtype dt,
                             const float* logits, int T, int top_k, void* out, void* ws,
                             size_t ws_bytes, void* stream) {
  return exl3_moe_forward_ex(layer, x, dt, logits, T, top_k, nullptr, out, EXL3_PATH_AUTO, ws,
                             ws_bytes, stream);
}

exl3_status exl3_rmsnorm(const void* x, exl3_dtype dt, int T, int H, float eps, void* out,
                         void* stream) {
  if (dt != EXL3_F16 && dt != EXL3_BF16) return EXL3_ERR_ARG;
  if (T < 0 || H <= 0 || H % 4) return EXL3_ERR_SHAPE;
  if (T > 0 && (!x || !out || !aligned16(out))) return EXL3_ERR_ARG;
  if (launch_rmsnorm(x, dt == EXL3_BF16, T, H, eps, out, static_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return EXL3_ERR_CUDA;
  return EXL3_OK;
}

exl3_status exl3_layer_set_stage_events(exl3_layer_t* layer, void* const* events, int n_events) {
  if (!layer) return EXL3_ERR_ARG;
  if (!events) {
    layer->has_ev = 0;
    return EXL3_OK;
  }
  if (n_events != EXL3_NUM_STAGE_EVENTS) return EXL3_ERR_ARG;
  for (int i = 0; i < EXL3_NUM_STAGE_EVENTS; i++) {
    if (!events[i]) return EXL3_ERR_ARG;
    layer->ev[i] = static_cast<cudaEvent_t>(events[i]);
  }
  layer->has_ev = 1;
  return EXL3_OK;
}

uint64_t exl3_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

exl3_status exl3_get_device_status(const void* ws, void* stream, int32_t* status) {
  if (!ws || !status) return EXL3_ERR_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return EXL3_ERR_CUDA;
  if (cudaMemcpy(status, ws, sizeof(int32_t), cudaMemcpyDeviceToHost) != cudaSuccess)
    return EXL3_ERR_CUDA;
  return *status ? EXL3_ERR_DEVICE : EXL3_OK;
}

}  // extern "C"
