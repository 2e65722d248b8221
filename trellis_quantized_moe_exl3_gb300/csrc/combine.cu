// Combine: y_t = sum_{j=0..k-1} r_{t,j} (fixed order) + shared(x_t)
// (+ residual), rounded once to the output dtype.  Atomic-free: the down
// projection wrote every pair row to its own slot (t, j).  Page "GLM-5.3
// Flash EXL3 for 2x DGX Sparks", section Cold prefill (E3): down + scatter.
// Also the RMSNorm used between stacked layers of a long prefill.
#include "common.cuh"
#include "internal.h"

namespace exl3 {

namespace {

__device__ __forceinline__ void store_act4(void* out, int bf16, size_t idx, float4 v) {
  if (bf16) {
    __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
    __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&a);
    u.y = *reinterpret_cast<uint32_t*>(&b);
    *reinterpret_cast<uint2*>(static_cast<uint16_t*>(out) + idx) = u;
  } else {
    __half2 a = __floats2half2_rn(v.x, v.y);
    __half2 b = __floats2half2_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&a);
    u.y = *reinterpret_cast<uint32_t*>(&b);
    *reinterpret_cast<uint2*>(static_cast<uint16_t*>(out) + idx) = u;
  }
}

// Pair j of token t takes part when its expert is in the call's range.
__device__ __forceinline__ bool in_shard(const int32_t* ids, size_t pair, Shard sh) {
  const int e = ids[pair];
  return e >= sh.e0 && e < sh.e1;
}

// The 4 outputs: rounded to the activation dtype, or (out_f32) the fp32 sum.
__device__ __forceinline__ void store_out4(void* out, int bf16, int f32, size_t idx, float4 v) {
  if (f32)
    *reinterpret_cast<float4*>(static_cast<float*>(out) + idx) = v;
  else
    store_act4(out, bf16, idx, v);
}

// One thread per group of 4 outputs, for unsplit pair rows: the k pair rows
// and the shared-expert partials are added in order.
__global__ void __launch_bounds__(256) combine_rows_kernel(const float* __restrict__ r, int T,
                                                           int k, int H, const int32_t* ids,
                                                           Shard sh,
                                                           const float* __restrict__ sp, int ns,
                                                           const void* __restrict__ resid,
                                                           void* __restrict__ out, int bf16,
                                                           int f32) {
  pdl_wait();
  const size_t n4 = (size_t)T * H / 4;
  for (size_t v = (size_t)blockIdx.x * blockDim.x + threadIdx.x; v < n4;
       v += (size_t)gridDim.x * blockDim.x) {
    const size_t t = v / (H / 4), o = (v % (H / 4)) * 4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < k; j++) {
      if (!in_shard(ids, t * k + j, sh)) continue;
      const float4 q = __ldcs(reinterpret_cast<const float4*>(r + (t * k + j) * H + o));
      acc.x += q.x; acc.y += q.y; acc.z += q.z; acc.w += q.w;
    }
    if (sp) {
      float4 s4 = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int s = 0; s < ns; s++) {
        const float4 q = *reinterpret_cast<const float4*>(sp + ((size_t)s * T + t) * H + o);
        s4.x += q.x; s4.y += q.y; s4.z += q.z; s4.w += q.w;
      }
      acc.x += s4.x; acc.y += s4.y; acc.z += s4.z; acc.w += s4.w;
    }
    if (resid) {
      acc.x += load_act(resid, bf16, t * H + o + 0);
      acc.y += load_act(resid, bf16, t * H + o + 1);
      acc.z += load_act(resid, bf16, t * H + o + 2);
      acc.w += load_act(resid, bf16, t * H + o + 3);
    }
    store_out4(out, bf16, f32, t * H + o, acc);
  }
}

// Eight lanes per group of 4 outputs: lane l of the octet adds the K-split
// partials of pairs j = l, l + 8 (splits in order) and the shared-expert
// partials s = l, l + 8, ... (in order); lane 0 then adds the eight lanes'
// sums in lane order, so the result is the same on every run.
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ r, int nr, int T,
                                                      int k, int H, const int32_t* ids, Shard sh,
                                                      const float* __restrict__ sp,
                                                      int ns, const void* __restrict__ resid,
                                                      void* __restrict__ out, int bf16, int f32) {
  pdl_wait();
  const int lane = threadIdx.x & 31, l8 = lane & 7, base = lane & 24;
  const size_t n4 = (size_t)T * H / 4;
  const size_t rstride = (size_t)T * k * H;  // one K-split slab of pair rows
  const size_t first = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) >> 3;
  const size_t step = ((size_t)gridDim.x * blockDim.x) >> 3;
  // every lane of a warp runs the same number of iterations (shuffles below)
  const size_t n_iter = (n4 + step - 1) / step;
  for (size_t it = 0; it < n_iter; it++) {
    const size_t v = first + it * step;
    const bool live = v < n4;
    const size_t t = live ? v / (H / 4) : 0, o = live ? (v % (H / 4)) * 4 : 0;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
    if (live) {
      for (int j = l8; j < k; j += 8) {
        if (!in_shard(ids, t * k + j, sh)) continue;
        const float* rp = r + (t * k + j) * H + o;
        float4 pr = *reinterpret_cast<const float4*>(rp);
#pragma unroll 8
        for (int q = 1; q < nr; q++) {
          const float4 w = *reinterpret_cast<const float4*>(rp + q * rstride);
          pr.x += w.x; pr.y += w.y; pr.z += w.z; pr.w += w.w;
        }
        a.x += pr.x; a.y += pr.y; a.z += pr.z; a.w += pr.w;
      }
      if (sp) {
#pragma unroll 4
        for (int s = l8; s < ns; s += 8) {
          const float4 w = *reinterpret_cast<const float4*>(sp + ((size_t)s * T + t) * H + o);
          b.x += w.x; b.y += w.y; b.z += w.z; b.w += w.w;
        }
      }
    }
    float4 acc = a, sh = b;
    for (int i = 1; i < 8; i++) {
      const int src = base + i;
      const float ax = __shfl_sync(0xffffffffu, a.x, src), ay = __shfl_sync(0xffffffffu, a.y, src);
      const float az = __shfl_sync(0xffffffffu, a.z, src), aw = __shfl_sync(0xffffffffu, a.w, src);
      const float bx = __shfl_sync(0xffffffffu, b.x, src), by = __shfl_sync(0xffffffffu, b.y, src);
      const float bz = __shfl_sync(0xffffffffu, b.z, src), bw = __shfl_sync(0xffffffffu, b.w, src);
      acc.x += ax; acc.y += ay; acc.z += az; acc.w += aw;
      sh.x += bx; sh.y += by; sh.z += bz; sh.w += bw;
    }
    if (live && l8 == 0) {
      acc.x += sh.x; acc.y += sh.y; acc.z += sh.z; acc.w += sh.w;
      if (resid) {
        acc.x += load_act(resid, bf16, t * H + o + 0);
        acc.y += load_act(resid, bf16, t * H + o + 1);
        acc.z += load_act(resid, bf16, t * H + o + 2);
        acc.w += load_act(resid, bf16, t * H + o + 3);
      }
      store_out4(out, bf16, f32, t * H + o, acc);
    }
  }
}

// out = round(y + residual), 4 outputs per thread.
__global__ void __launch_bounds__(256) round_output_kernel(const float* __restrict__ y, size_t n4,
                                                           const void* __restrict__ resid,
                                                           void* __restrict__ out, int bf16) {
  for (size_t v = (size_t)blockIdx.x * blockDim.x + threadIdx.x; v < n4;
       v += (size_t)gridDim.x * blockDim.x) {
    float4 a = reinterpret_cast<const float4*>(y)[v];
    if (resid) {
      a.x += load_act(resid, bf16, 4 * v + 0);
      a.y += load_act(resid, bf16, 4 * v + 1);
      a.z += load_act(resid, bf16, 4 * v + 2);
      a.w += load_act(resid, bf16, 4 * v + 3);
    }
    store_act4(out, bf16, 4 * v, a);
  }
}

__global__ void __launch_bounds__(256) rmsnorm_kernel(const void* __restrict__ x, int bf16, int H,
                                                      float eps, void* __restrict__ out) {
  pdl_wait();
  __shared__ float s_w[32];
  const size_t t = blockIdx.x;
  float ss = 0.0f;
  for (int i = threadIdx.x; i < H; i += blockDim.x) {
    const float v = load_act(x, bf16, t * H + i);
    ss = fmaf(v, v, ss);
  }
  for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  if ((threadIdx.x & 31) == 0) s_w[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.0f;
  for (int w = 0; w < (int)(blockDim.x >> 5); w++) tot += s_w[w];
  const float inv = 1.0f / sqrtf(tot / (float)H + eps);
  __syncthreads();  // all reads of x done before any in-place write
  for (int i = threadIdx.x * 4; i < H; i += blockDim.x * 4) {
    float4 v;
    v.x = load_act(x, bf16, t * H + i) * inv;
    v.y = load_act(x, bf16, t * H + i + 1) * inv;
    v.z = load_act(x, bf16, t * H + i + 2) * inv;
    v.w = load_act(x, bf16, t * H + i + 3) * inv;
    store_act4(out, bf16, t * H + i, v);
  }
}

}  // namespace

cudaError_t launch_combine(const float* r, int r_splits, int T, int top_k, int H,
                           const int32_t* ids, Shard sh, const float* shared_part,
                           int shared_splits, const void* residual, void* out, int out_bf16,
                           int out_f32, cudaStream_t st) {
  const size_t n4 = (size_t)T * H / 4;
  cudaError_t err;
  if (r_splits == 1) {
    size_t blocks = (n4 + 255) / 256;
    if (blocks > 152 * 16) blocks = 152 * 16;
    if (blocks < 1) blocks = 1;
    err = launch_pdl(combine_rows_kernel, dim3((unsigned)blocks), dim3(256), 0, st, r, T, top_k, H,
                     ids, sh, shared_part, shared_splits, residual, out, out_bf16, out_f32);
  } else {
    size_t blocks = (n4 * 8 + 255) / 256;
    if (blocks > 152 * 16) blocks = 152 * 16;
    if (blocks < 1) blocks = 1;
    err = launch_pdl(combine_kernel, dim3((unsigned)blocks), dim3(256), 0, st, r, r_splits, T,
                     top_k, H, ids, sh, shared_part, shared_splits, residual, out, out_bf16,
                     out_f32);
  }
  note_launches(1);
  return err;
}

cudaError_t launch_round_output(const float* y, int T, int H, const void* residual, void* out,
                                int out_bf16, cudaStream_t st) {
  const size_t n4 = (size_t)T * H / 4;
  if (n4 == 0) return cudaSuccess;
  size_t blocks = (n4 + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  const cudaError_t err = launch_pdl(round_output_kernel, dim3((unsigned)blocks), dim3(256), 0, st,
                                     y, n4, residual, out, out_bf16);
  note_launches(1);
  return err;
}

cudaError_t launch_rmsnorm(const void* x, int bf16, int T, int H, float eps, void* out,
                           cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  const cudaError_t err = launch_pdl(rmsnorm_kernel, dim3(T), dim3(256), 0, st, x, bf16, H, eps, out);
  note_launches(1);
  return err;
}

}  // namespace exl3
