// Shared expert: an unquantized fp16 SwiGLU MLP of the routed experts' shape,
// added with weight 1 (page "GLM-5.3-Flash · exlr8 (K2/K3/K4)", intro: one
// shared expert per MoE layer; page "GLM-5.3-Flash EXL3 (~2.1 bpw, SM70 tile
// order)", Recipe: shared experts kept FP16).
//
// HBM-bound GEMV: each thread streams 8 consecutive outputs of one weight row
// (16-byte loads, a warp covers 512 contiguous bytes) over a slice of
// kSharedKPer input rows, for up to 8 tokens at a time, and writes a partial
// sum per slice.  The slices are added in a fixed order by the consumer (the
// down projection's prologue, then the combine), so the result is
// deterministic without atomics.
#include "common.cuh"
#include "internal.h"

namespace exl3 {

namespace {

constexpr int kTT = 8;  // tokens per pass

// mode 0: input rows are x (fp16/bf16) [T][in]
// mode 1: input h = silu(sum_s pg[s]) * sum_s pu[s], pg/pu: [nsplit][T][in] fp32
__global__ void __launch_bounds__(128) shared_gemv_kernel(const uint16_t* __restrict__ W, int in,
                                                          int out, int mode,
                                                          const void* __restrict__ x, int x_bf16,
                                                          const float* __restrict__ pg,
                                                          const float* __restrict__ pu,
                                                          int nsplit_in, int T,
                                                          float* __restrict__ part) {
  __shared__ float s_in[kTT][kSharedKPer];
  const int split = blockIdx.y;
  const int k0 = split * kSharedKPer;
  const int t0 = blockIdx.z * kTT;
  const int nt = min(kTT, T - t0);
  for (int v = threadIdx.x; v < kTT * kSharedKPer; v += blockDim.x) {
    const int tt = v / kSharedKPer, kk = v % kSharedKPer;
    float val = 0.0f;
    if (tt < nt) {
      const int t = t0 + tt;
      if (mode == 0) {
        val = load_act(x, x_bf16, (size_t)t * in + k0 + kk);
      } else {
        float g = 0.0f, u = 0.0f;
        for (int s = 0; s < nsplit_in; s++) {
          g += pg[((size_t)s * T + t) * in + k0 + kk];
          u += pu[((size_t)s * T + t) * in + k0 + kk];
        }
        val = silu_f(g) * u;
      }
    }
    s_in[tt][kk] = val;
  }
  __syncthreads();
  const int o0 = (blockIdx.x * blockDim.x + threadIdx.x) * 8;
  if (o0 >= out) return;
  float acc[kTT][8];
#pragma unroll
  for (int tt = 0; tt < kTT; tt++)
#pragma unroll
    for (int q = 0; q < 8; q++) acc[tt][q] = 0.0f;
  const uint16_t* wp = W + (size_t)k0 * out + o0;
#pragma unroll 4
  for (int kk = 0; kk < kSharedKPer; kk++) {
    uint4 raw;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(raw.x), "=r"(raw.y), "=r"(raw.z), "=r"(raw.w)
                 : "l"(wp + (size_t)kk * out));
    const uint32_t rr[4] = {raw.x, raw.y, raw.z, raw.w};
    float wf[8];
#pragma unroll
    for (int q = 0; q < 4; q++) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&rr[q]));
      wf[2 * q] = f.x;
      wf[2 * q + 1] = f.y;
    }
#pragma unroll
    for (int tt = 0; tt < kTT; tt++) {
      const float xv = s_in[tt][kk];
#pragma unroll
      for (int q = 0; q < 8; q++) acc[tt][q] = fmaf(xv, wf[q], acc[tt][q]);
    }
  }
  for (int tt = 0; tt < nt; tt++) {
    float* dst = part + ((size_t)split * T + t0 + tt) * out + o0;
    reinterpret_cast<float4*>(dst)[0] = make_float4(acc[tt][0], acc[tt][1], acc[tt][2], acc[tt][3]);
    reinterpret_cast<float4*>(dst)[1] = make_float4(acc[tt][4], acc[tt][5], acc[tt][6], acc[tt][7]);
  }
}

}  // namespace

size_t shared_scratch_bytes(int T, int H, int I) {
  const size_t gu = (size_t)2 * (H / kSharedKPer) * T * I * 4;
  const size_t d = (size_t)(I / kSharedKPer) * T * H * 4;
  return ((gu + 255) & ~(size_t)255) + ((d + 255) & ~(size_t)255);
}

// part_gu: [2][H/kper][T][I]; part_d: [I/kper][T][H]
cudaError_t launch_shared(const LayerView& L, const void* x, int x_bf16, int T, float* part_gu,
                          float* part_d, cudaStream_t st) {
  const int sh = L.H / kSharedKPer, si = L.I / kSharedKPer;
  const int tz = (T + kTT - 1) / kTT;
  float* pg = part_gu;
  float* pu = part_gu + (size_t)sh * T * L.I;
  dim3 g1((L.I / 8 + 127) / 128, sh, tz);
  shared_gemv_kernel<<<g1, 128, 0, st>>>(L.shared_w[0], L.H, L.I, 0, x, x_bf16, nullptr, nullptr,
                                         0, T, pg);
  shared_gemv_kernel<<<g1, 128, 0, st>>>(L.shared_w[1], L.H, L.I, 0, x, x_bf16, nullptr, nullptr,
                                         0, T, pu);
  dim3 g2((L.H / 8 + 127) / 128, si, tz);
  shared_gemv_kernel<<<g2, 128, 0, st>>>(L.shared_w[2], L.I, L.H, 1, nullptr, 0, pg, pu, sh, T,
                                         part_d);
  note_launches(3);
  return cudaGetLastError();
}

}  // namespace exl3
