// Shared expert: an unquantized fp16 SwiGLU MLP of the routed experts' shape,
// added with weight 1 (page "GLM-5.3-Flash · exlr8 (K2/K3/K4)", intro: one
// shared expert per MoE layer; page "GLM-5.3-Flash EXL3 (~2.1 bpw, SM70 tile
// order)", Recipe: shared experts kept FP16).
//
// For decode-sized T this is a stream over 3 x H x I fp16 weights, bound by
// HBM bandwidth.  One CTA = 8 warps on the same 256 outputs (a lane owns 8
// consecutive outputs, so a warp reads 512 contiguous bytes of a weight row),
// each warp on its own 16 rows of the CTA's 128-row input slice, all 16 row
// loads of a lane in flight before the first FMA; the 8 warps' sums are added
// in shared memory, warp by warp, into the CTA's K-split slab.
//   gate/up launch: partial sums [proj][split][T][I];
//   h launch: h = silu(sum of gate slabs) * (sum of up slabs), slabs in order;
//   down launch: partial sums [split][T][H] that the combine adds in order.
// Tokens are processed in passes of up to 8 (blockIdx.z); the result does not
// depend on scheduling and no atomics are used.
#include "common.cuh"
#include "internal.h"

namespace exl3 {

namespace {

constexpr int kSWarps = 8;
constexpr int kSThreads = kSWarps * 32;
constexpr int kSOut = 256;    // outputs per CTA
constexpr int kSBatch = 16;   // rows a lane has in flight
constexpr int kSPass = 8;     // tokens per pass
constexpr int kSRows = kSWarps * kSBatch;  // input rows per CTA (128)

struct SharedParams {
  const uint16_t* w[2];  // [in][out] fp16 (gate, up) or (down)
  int in, out, T;
  int nproj;             // 2: gate and up, 1: down
  const void* x;         // input rows [T][in]: activations (fp16/bf16) ...
  int x_bf16;
  const float* h;        // ... or fp32 h (down)
  float* part;           // [nproj][in / 128][T][out]
};

__device__ __forceinline__ void f16x2_to_f32(uint32_t u, float& lo, float& hi) {
  lo = __half2float(__ushort_as_half((unsigned short)(u & 0xFFFFu)));
  hi = __half2float(__ushort_as_half((unsigned short)(u >> 16)));
}

__device__ __forceinline__ void load_rows(uint4 (&raw)[kSBatch], const uint16_t* wp, int out,
                                          bool ok) {
#pragma unroll
  for (int r = 0; r < kSBatch; r++) {
    raw[r] = make_uint4(0, 0, 0, 0);
    if (ok)
      asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                   : "=r"(raw[r].x), "=r"(raw[r].y), "=r"(raw[r].z), "=r"(raw[r].w)
                   : "l"(wp + (size_t)r * out));
  }
}

template <int NT>
__device__ __forceinline__ void fma_rows(float (&acc)[NT][8], const uint4 (&raw)[kSBatch],
                                         const float* s_in, int ld, int row0) {
#pragma unroll
  for (int r = 0; r < kSBatch; r++) {
    float wf[8];
    f16x2_to_f32(raw[r].x, wf[0], wf[1]);
    f16x2_to_f32(raw[r].y, wf[2], wf[3]);
    f16x2_to_f32(raw[r].z, wf[4], wf[5]);
    f16x2_to_f32(raw[r].w, wf[6], wf[7]);
#pragma unroll
    for (int t = 0; t < NT; t++) {
      const float xv = s_in[t * ld + row0 + r];
#pragma unroll
      for (int q = 0; q < 8; q++) acc[t][q] = fmaf(xv, wf[q], acc[t][q]);
    }
  }
}

template <int NT>
__global__ void __launch_bounds__(kSThreads, 2) shared_gemv_kernel(SharedParams p) {
  extern __shared__ __align__(16) float s_red[];  // [kSWarps][NT][kSOut]
  __shared__ float s_in[NT * kSRows];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int chunk = blockIdx.x, split = blockIdx.y;
  const int pj = blockIdx.z % p.nproj, pass = blockIdx.z / p.nproj;
  const int t0 = pass * kSPass;
  const int nt = min(NT, p.T - t0);
  const int k0 = split * kSRows;

  // the weight rows go out before the inputs are staged
  // (out is a multiple of 128: the last chunk may be half full)
  const bool lane_ok = chunk * kSOut + lane * 8 < p.out;
  const uint16_t* wp =
      (pj ? p.w[1] : p.w[0]) + (size_t)(k0 + warp * kSBatch) * p.out + chunk * kSOut + lane * 8;
  uint4 raw[kSBatch];
  load_rows(raw, wp, p.out, lane_ok);

  // the inputs (h) and the partial sums are the predecessors' business
  pdl_wait();
  for (int v = threadIdx.x; v < NT * kSRows; v += kSThreads) {
    const int tt = v / kSRows, kk = v % kSRows;
    float val = 0.0f;
    if (tt < nt) {
      const size_t idx = (size_t)(t0 + tt) * p.in + k0 + kk;
      val = p.h ? p.h[idx] : load_act(p.x, p.x_bf16, idx);
    }
    s_in[v] = val;
  }
  __syncthreads();

  float acc[NT][8];
#pragma unroll
  for (int t = 0; t < NT; t++)
#pragma unroll
    for (int q = 0; q < 8; q++) acc[t][q] = 0.0f;
  fma_rows<NT>(acc, raw, s_in, kSRows, warp * kSBatch);
#pragma unroll
  for (int t = 0; t < NT; t++) {
    float4* d = reinterpret_cast<float4*>(s_red + ((size_t)warp * NT + t) * kSOut + lane * 8);
    d[0] = make_float4(acc[t][0], acc[t][1], acc[t][2], acc[t][3]);
    d[1] = make_float4(acc[t][4], acc[t][5], acc[t][6], acc[t][7]);
  }
  __syncthreads();

  // CTA sum in warp order, one (token, output) per thread and step
  const int nsplit = p.in / kSRows;
  float* part = p.part + (size_t)pj * nsplit * p.T * p.out;
  const int nout = min(kSOut, p.out - chunk * kSOut);
  for (int v = threadIdx.x; v < nt * kSOut; v += kSThreads) {
    const int t = v / kSOut, o = v % kSOut;
    if (o >= nout) continue;
    float s = 0.0f;
#pragma unroll
    for (int w = 0; w < kSWarps; w++) s += s_red[((size_t)w * NT + t) * kSOut + o];
    part[((size_t)split * p.T + t0 + t) * p.out + chunk * kSOut + o] = s;
  }
}

// h[t][o] = silu(sum_s gate[s][t][o]) * sum_s up[s][t][o], splits in order.
__global__ void __launch_bounds__(256) shared_h_kernel(const float* __restrict__ part, int nsplit,
                                                       int T, int I, float* __restrict__ h) {
  pdl_wait();
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (size_t)T * I) return;
  const size_t slab = (size_t)T * I;
  const float* pg = part + i;
  const float* pu = part + (size_t)nsplit * slab + i;
  float g = 0.0f, u = 0.0f;
#pragma unroll 8
  for (int s = 0; s < nsplit; s++) {
    g += pg[s * slab];
    u += pu[s * slab];
  }
  h[i] = silu_f(g) * u;
}

template <int NT>
cudaError_t launch_nt(const SharedParams& sp, dim3 grid, cudaStream_t st) {
  const int smem = kSWarps * NT * kSOut * 4;
  static bool attr = false;
  if (!attr) {
    const cudaError_t e = cudaFuncSetAttribute(shared_gemv_kernel<NT>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  const cudaError_t err = launch_pdl(shared_gemv_kernel<NT>, grid, dim3(kSThreads), smem, st, sp);
  note_launches(1);
  return err;
}

cudaError_t launch_sg(const SharedParams& sp, dim3 grid, cudaStream_t st) {
  const int nt = sp.T < kSPass ? sp.T : kSPass;
  if (nt <= 1) return launch_nt<1>(sp, grid, st);
  if (nt <= 2) return launch_nt<2>(sp, grid, st);
  if (nt <= 4) return launch_nt<4>(sp, grid, st);
  return launch_nt<8>(sp, grid, st);
}

struct SharedLayout {
  size_t part_gu, h, part_d, total;
};

SharedLayout shared_layout(int T, int H, int I) {
  auto al = [](size_t b) { return (b + 255) & ~(size_t)255; };
  SharedLayout s{};
  size_t o = 0;
  s.part_gu = o; o += al((size_t)2 * (H / kSRows) * T * I * 4);
  s.h = o; o += al((size_t)T * I * 4);
  s.part_d = o; o += al((size_t)(I / kSRows) * T * H * 4);
  s.total = o;
  return s;
}

}  // namespace

size_t shared_scratch_bytes(int T, int H, int I) { return shared_layout(T, H, I).total; }

cudaError_t launch_shared(const LayerView& L, const void* x, int x_bf16, int T, void* scratch,
                          const float** part_d, int* nsplit_d, cudaStream_t st) {
  const SharedLayout s = shared_layout(T, L.H, L.I);
  char* b = static_cast<char*>(scratch);
  const int passes = (T + kSPass - 1) / kSPass;
  const int chunks_i = (L.I + kSOut - 1) / kSOut, chunks_h = (L.H + kSOut - 1) / kSOut;
  cudaError_t err;
  SharedParams gu{};
  gu.w[0] = L.shared_w[0]; gu.w[1] = L.shared_w[1];
  gu.in = L.H; gu.out = L.I; gu.T = T; gu.nproj = 2;
  gu.x = x; gu.x_bf16 = x_bf16;
  gu.part = reinterpret_cast<float*>(b + s.part_gu);
  if ((err = launch_sg(gu, dim3(chunks_i, L.H / kSRows, 2 * passes), st)) != cudaSuccess) return err;
  float* h = reinterpret_cast<float*>(b + s.h);
  const size_t nh = (size_t)T * L.I;
  err = launch_pdl(shared_h_kernel, dim3((unsigned)((nh + 255) / 256)), dim3(256), 0, st, gu.part,
                   L.H / kSRows, T, L.I, h);
  note_launches(1);
  if (err != cudaSuccess) return err;
  SharedParams dn{};
  dn.w[0] = L.shared_w[2];
  dn.in = L.I; dn.out = L.H; dn.T = T; dn.nproj = 1;
  dn.h = h;
  dn.part = reinterpret_cast<float*>(b + s.part_d);
  if ((err = launch_sg(dn, dim3(chunks_h, L.I / kSRows, passes), st)) != cudaSuccess) return err;
  *part_d = dn.part;
  *nsplit_d = L.I / kSRows;
  return cudaSuccess;
}

}  // namespace exl3
