// Grouped GEMV path for decode-sized steps (a few tokens per expert).
//
// Page "GLM-5.3-Flash EXL3 (~2.1 bpw, SM70 tile order)", Running it: the
// expert kernels decode the trellis inside the matmul; Speed: per-lane window
// loads of the strip-major tiles.  Page "GLM-5.3 Flash EXL3 for 2x DGX
// Sparks", section Cold prefill (E3): gather, gate/up + SwiGLU, down +
// scatter, driven by device-side segment tables.
//
// Work item = (active expert, 128-output strip, group of 8 tokens).  Each
// warp of a CTA takes every W-th 16-input block; per block it streams the 8
// consecutive tiles of the strip with one coalesced load per lane (8K bytes
// per lane), decodes its 64 weights in registers (the 16-K bit overlap comes
// from the next lane of the quad by shuffle) and feeds them to mma.m16n8k16
// with the K dimension doubled: the A register of weight (o, i) is the
// codebook's {a, b} fp16 pair itself and the B register holds {x_i, x_i}, so
// the tensor core forms (a + b) * x_i without a separate add.  (The exact sum
// a + b differs from the format's fp16(a + b) by at most half an fp16 ulp,
// far inside the layer tolerance; with the E4M3 rule the rounded value is
// formed first and placed as {v, 0}.)  Partial sums of the W warps are added
// in a fixed order in shared memory; no atomics anywhere.
//
// Activations enter as fp16 with a power-of-two scale per (pair, projection)
// chosen from the row's max |x * suh| (undone in the epilogue), so the fp16
// operand never overflows whatever the input magnitude.
#include "common.cuh"
#include "internal.h"

namespace exl3 {

namespace {

constexpr int kW = 4;  // warps per CTA

__device__ __forceinline__ float block_max(float v, float* s_tmp) {
  for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  __syncthreads();
  if (lane == 0) s_tmp[wid] = v;
  __syncthreads();
  float r = 0.0f;
  for (int w = 0; w < nw; w++) r = fmaxf(r, s_tmp[w]);
  return r;
}

__device__ __forceinline__ uint32_t dup_f16(float v) {
  const uint32_t b = __half_as_ushort(__float2half_rn(v));
  return b | (b << 16);
}

// Slot of input idx inside its 16-block: lane c reads slots 4c..4c+3, which
// hold inputs c, c+4, c+8, c+12.
__device__ __forceinline__ int perm_slot(int idx) {
  const int r = idx & 15;
  return 4 * (r & 3) + (r >> 2);
}

// x rows of the pairs in segment order, times suh of gate and up, scaled.
__global__ void __launch_bounds__(256) gather_xs_kernel(const void* __restrict__ x, int x_bf16,
                                                        int H, int k, const int32_t* seg_pairs,
                                                        const int32_t* ids,
                                                        const uint16_t* __restrict__ suh_g,
                                                        const uint16_t* __restrict__ suh_u,
                                                        uint32_t* __restrict__ xs,
                                                        float* __restrict__ xs_inv) {
  __shared__ float s_tmp[32];
  const int pos = blockIdx.x;
  const int p = seg_pairs[pos];
  const int t = p / k, e = ids[p];
  const uint16_t* sg = suh_g + (size_t)e * H;
  const uint16_t* su = suh_u + (size_t)e * H;
  float ag = 0.0f, au = 0.0f;
  for (int idx = threadIdx.x; idx < H; idx += blockDim.x) {
    const float xv = load_act(x, x_bf16, (size_t)t * H + idx);
    ag = fmaxf(ag, fabsf(xv * __half2float(__ushort_as_half(sg[idx]))));
    au = fmaxf(au, fabsf(xv * __half2float(__ushort_as_half(su[idx]))));
  }
  ag = block_max(ag, s_tmp);
  au = block_max(au, s_tmp);
  const int eg = fp16_scale_exp(ag), eu = fp16_scale_exp(au);
  const float scg = ldexpf(1.0f, eg), scu = ldexpf(1.0f, eu);
  uint32_t* og = xs + (size_t)pos * 2 * H;
  uint32_t* ou = og + H;
  for (int idx = threadIdx.x; idx < H; idx += blockDim.x) {
    const float xv = load_act(x, x_bf16, (size_t)t * H + idx);
    const int dst = (idx & ~15) + perm_slot(idx);
    og[dst] = dup_f16(xv * __half2float(__ushort_as_half(sg[idx])) * scg);
    ou[dst] = dup_f16(xv * __half2float(__ushort_as_half(su[idx])) * scu);
  }
  if (threadIdx.x == 0) {
    xs_inv[2 * pos] = ldexpf(1.0f, -eg);
    xs_inv[2 * pos + 1] = ldexpf(1.0f, -eu);
  }
}

// h rows (pair-sorted) times suh of down, scaled, permuted, duplicated.
__global__ void __launch_bounds__(256) prep_down_kernel(const float* __restrict__ h, int I,
                                                        const int32_t* seg_pairs,
                                                        const int32_t* ids,
                                                        const uint16_t* __restrict__ suh_d,
                                                        uint32_t* __restrict__ xs,
                                                        float* __restrict__ xs_inv) {
  __shared__ float s_tmp[32];
  const int pos = blockIdx.x;
  const int e = ids[seg_pairs[pos]];
  const uint16_t* sd = suh_d + (size_t)e * I;
  const float* hr = h + (size_t)pos * I;
  float am = 0.0f;
  for (int idx = threadIdx.x; idx < I; idx += blockDim.x)
    am = fmaxf(am, fabsf(hr[idx] * __half2float(__ushort_as_half(sd[idx]))));
  am = block_max(am, s_tmp);
  const int ex = fp16_scale_exp(am);
  const float sc = ldexpf(1.0f, ex);
  uint32_t* o = xs + (size_t)pos * I;
  for (int idx = threadIdx.x; idx < I; idx += blockDim.x)
    o[(idx & ~15) + perm_slot(idx)] = dup_f16(hr[idx] * __half2float(__ushort_as_half(sd[idx])) * sc);
  if (threadIdx.x == 0) xs_inv[pos] = ldexpf(1.0f, -ex);
}

template <int K, int FP8>
__device__ __forceinline__ void decode_mma(const LaneWords<K>& lw, const uint4& b,
                                           float (&acc)[8][4], uint32_t mult) {
#pragma unroll
  for (int r0 = 0; r0 < 8; r0++) {
#pragma unroll
    for (int hf = 0; hf < 2; hf++) {
      const int u = 8 * r0 + 4 * hf;
      uint32_t a0, a1, a2, a3;
      const uint32_t m0 = mcg_halves(lane_state<K>(lw, u + 0), mult);
      const uint32_t m1 = mcg_halves(lane_state<K>(lw, u + 1), mult);
      const uint32_t m2 = mcg_halves(lane_state<K>(lw, u + 2), mult);
      const uint32_t m3 = mcg_halves(lane_state<K>(lw, u + 3), mult);
      if (!FP8) {
        a0 = m0; a1 = m1; a2 = m2; a3 = m3;
      } else {
        const uint32_t v01 = e4m3_round2(sum_halves2(m0, m1));
        const uint32_t v23 = e4m3_round2(sum_halves2(m2, m3));
        a0 = v01 & 0xFFFFu; a1 = v01 >> 16; a2 = v23 & 0xFFFFu; a3 = v23 >> 16;
      }
      mma_f16_16816(acc[r0], a0, a1, a2, a3, hf ? b.z : b.x, hf ? b.w : b.y);
    }
  }
}

struct GemvParams {
  const uint16_t* codes[2];
  size_t stride[2];       // uint16 words per expert
  int in, out;
  uint32_t mult;
  const uint16_t* svh[2]; // [E][out]
  const uint32_t* xs;     // [pos][NPROJ][in] fp16x2 permuted
  const float* xs_inv;    // [pos][NPROJ]
  const int32_t* seg_offsets;
  const int32_t* active;
  const int32_t* seg_pairs;
  const float* wts;       // router weights by pair id
  float* h_out;           // NPROJ == 2: [pos][out]
  float* r_out;           // NPROJ == 1: [pair id][out]
};

__device__ __forceinline__ uint4 ld_b(const uint32_t* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

template <int K, int FP8, int NPROJ>
__global__ void __launch_bounds__(kW * 32) gemv_kernel(GemvParams p) {
  extern __shared__ float s_red[];  // [kW][NPROJ][1024]
  const int strips = p.out / 128;
  const int slot = blockIdx.x / strips, s = blockIdx.x % strips;
  if (slot >= p.active[0]) return;
  const int e = p.active[1 + slot];
  const int seg0 = p.seg_offsets[e], seg1 = p.seg_offsets[e + 1];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, g = lane >> 2, c = lane & 3;
  const int nblk = p.in / 16;
  const size_t row_words = (size_t)(p.out / 16) * 16 * K;
  const uint16_t* cbase[NPROJ];
#pragma unroll
  for (int pj = 0; pj < NPROJ; pj++)
    cbase[pj] = p.codes[pj] + p.stride[pj] * e + (size_t)8 * s * 16 * K + lane * 4 * K;

  for (int tg0 = seg0; tg0 < seg1; tg0 += 8) {
    float acc[NPROJ][8][4];
#pragma unroll
    for (int pj = 0; pj < NPROJ; pj++)
#pragma unroll
      for (int r = 0; r < 8; r++)
#pragma unroll
        for (int d = 0; d < 4; d++) acc[pj][r][d] = 0.0f;
    const int bpos = tg0 + g;
    const bool bvalid = bpos < seg1;
    const uint32_t* xrow[NPROJ];
#pragma unroll
    for (int pj = 0; pj < NPROJ; pj++)
      xrow[pj] = p.xs + ((size_t)(bvalid ? bpos : seg0) * NPROJ + pj) * p.in + 4 * c;

    LaneWords<K> cur[NPROJ], nxt[NPROJ];
    uint4 cb[NPROJ], nb[NPROJ];
    int i = warp;
    if (i < nblk) {
#pragma unroll
      for (int pj = 0; pj < NPROJ; pj++) {
        load_lane_words<K>(cur[pj], cbase[pj] + (size_t)i * row_words);
        cb[pj] = bvalid ? ld_b(xrow[pj] + i * 16) : make_uint4(0, 0, 0, 0);
      }
    }
    for (; i < nblk; i += kW) {
      const int inext = i + kW;
      if (inext < nblk) {
#pragma unroll
        for (int pj = 0; pj < NPROJ; pj++) {
          load_lane_words<K>(nxt[pj], cbase[pj] + (size_t)inext * row_words);
          nb[pj] = bvalid ? ld_b(xrow[pj] + inext * 16) : make_uint4(0, 0, 0, 0);
        }
      }
#pragma unroll
      for (int pj = 0; pj < NPROJ; pj++) {
        fetch_neighbour<K>(cur[pj]);
        decode_mma<K, FP8>(cur[pj], cb[pj], acc[pj], p.mult);
      }
#pragma unroll
      for (int pj = 0; pj < NPROJ; pj++) {
        cur[pj] = nxt[pj];
        cb[pj] = nb[pj];
      }
    }
    __syncthreads();  // the previous group's epilogue has finished with s_red
    float* my = s_red + (size_t)warp * NPROJ * 1024;
#pragma unroll
    for (int pj = 0; pj < NPROJ; pj++)
#pragma unroll
      for (int r = 0; r < 8; r++)
#pragma unroll
        for (int d = 0; d < 4; d++) my[pj * 1024 + (r * 32 + lane) * 4 + d] = acc[pj][r][d];
    __syncthreads();
    for (int v = threadIdx.x; v < 1024; v += blockDim.x) {
      float sum[NPROJ];
#pragma unroll
      for (int pj = 0; pj < NPROJ; pj++) sum[pj] = 0.0f;
      for (int w = 0; w < kW; w++)
#pragma unroll
        for (int pj = 0; pj < NPROJ; pj++) sum[pj] += s_red[((size_t)w * NPROJ + pj) * 1024 + v];
      const int r0 = v >> 7, ln = (v >> 2) & 31, d = v & 3;
      const int o = 16 * (8 * s + (ln >> 2)) + r0 + 8 * (d >> 1);
      const int pos = tg0 + 2 * (ln & 3) + (d & 1);
      if (pos < seg1) {
        if constexpr (NPROJ == 2) {
          const float G = sum[0] * p.xs_inv[2 * pos] *
                          __half2float(__ushort_as_half(p.svh[0][(size_t)e * p.out + o]));
          const float U = sum[1] * p.xs_inv[2 * pos + 1] *
                          __half2float(__ushort_as_half(p.svh[1][(size_t)e * p.out + o]));
          p.h_out[(size_t)pos * p.out + o] = silu_f(G) * U;
        } else {
          const int pid = p.seg_pairs[pos];
          p.r_out[(size_t)pid * p.out + o] =
              sum[0] * p.xs_inv[pos] *
              __half2float(__ushort_as_half(p.svh[0][(size_t)e * p.out + o])) * p.wts[pid];
        }
      }
    }
  }
}

template <int K, int FP8, int NPROJ>
cudaError_t launch_gemv(const GemvParams& gp, int grid, cudaStream_t st) {
  const size_t smem = (size_t)kW * NPROJ * 1024 * sizeof(float);
  gemv_kernel<K, FP8, NPROJ><<<grid, kW * 32, smem, st>>>(gp);
  note_launches(1);
  return cudaGetLastError();
}

template <int NPROJ>
cudaError_t dispatch_gemv(int K, int fp8, const GemvParams& gp, int grid, cudaStream_t st) {
  if (fp8) {
    if (K == 2) return launch_gemv<2, 1, NPROJ>(gp, grid, st);
    if (K == 3) return launch_gemv<3, 1, NPROJ>(gp, grid, st);
    return launch_gemv<4, 1, NPROJ>(gp, grid, st);
  }
  if (K == 2) return launch_gemv<2, 0, NPROJ>(gp, grid, st);
  if (K == 3) return launch_gemv<3, 0, NPROJ>(gp, grid, st);
  return launch_gemv<4, 0, NPROJ>(gp, grid, st);
}

static size_t al(size_t b) { return (b + 255) & ~(size_t)255; }

}  // namespace

size_t gemv_scratch_bytes(int T, int top_k, int H, int I) {
  const size_t P = (size_t)T * top_k;
  return al(P * 2 * H * 4) + al(P * 2 * 4) + al(P * I * 4) + al(P * I * 4) + al(P * 4) +
         al(P * H * 4);
}

void gemv_carve(void* ws, int T, int top_k, int H, int I, GemvBuffers* gb) {
  const size_t P = (size_t)T * top_k;
  char* q = static_cast<char*>(ws);
  gb->xs_gu = reinterpret_cast<uint32_t*>(q); q += al(P * 2 * H * 4);
  gb->xs_gu_inv = reinterpret_cast<float*>(q); q += al(P * 2 * 4);
  gb->h = reinterpret_cast<float*>(q); q += al(P * I * 4);
  gb->xs_d = reinterpret_cast<uint32_t*>(q); q += al(P * I * 4);
  gb->xs_d_inv = reinterpret_cast<float*>(q); q += al(P * 4);
  gb->r = reinterpret_cast<float*>(q);
}

cudaError_t launch_moe_gemv(const LayerView& L, const void* x, int x_bf16, int T, int top_k,
                            const RouteBuffers& rb, const GemvBuffers& gb, const cudaEvent_t* ev,
                            cudaStream_t st) {
  auto rec = [&](int i) {
    if (ev && ev[i]) record_stage_event(ev[i], st);
  };
  const int P = T * top_k;
  const int slots = P < L.E ? P : L.E;
  cudaError_t err;
  gather_xs_kernel<<<P, 256, 0, st>>>(x, x_bf16, L.H, top_k, rb.seg_pairs, rb.ids, L.suh[0],
                                      L.suh[1], gb.xs_gu, gb.xs_gu_inv);
  note_launches(1);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  rec(2);

  GemvParams gu{};
  gu.codes[0] = L.codes[0]; gu.codes[1] = L.codes[1];
  gu.stride[0] = L.code_stride[0]; gu.stride[1] = L.code_stride[1];
  gu.in = L.H; gu.out = L.I; gu.mult = L.mult;
  gu.svh[0] = L.svh[0]; gu.svh[1] = L.svh[1];
  gu.xs = gb.xs_gu; gu.xs_inv = gb.xs_gu_inv;
  gu.seg_offsets = rb.seg_offsets; gu.active = rb.active; gu.seg_pairs = rb.seg_pairs;
  gu.wts = rb.w; gu.h_out = gb.h;
  // gate and up share one launch, so they must share a width
  if (L.K[0] != L.K[1]) return cudaErrorInvalidValue;
  if ((err = dispatch_gemv<2>(L.K[0], L.fp8, gu, slots * (L.I / 128), st)) != cudaSuccess)
    return err;
  rec(3);

  prep_down_kernel<<<P, 256, 0, st>>>(gb.h, L.I, rb.seg_pairs, rb.ids, L.suh[2], gb.xs_d,
                                      gb.xs_d_inv);
  note_launches(1);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  rec(4);

  GemvParams dn{};
  dn.codes[0] = L.codes[2]; dn.stride[0] = L.code_stride[2];
  dn.in = L.I; dn.out = L.H; dn.mult = L.mult;
  dn.svh[0] = L.svh[2];
  dn.xs = gb.xs_d; dn.xs_inv = gb.xs_d_inv;
  dn.seg_offsets = rb.seg_offsets; dn.active = rb.active; dn.seg_pairs = rb.seg_pairs;
  dn.wts = rb.w; dn.r_out = gb.r;
  err = dispatch_gemv<1>(L.K[2], L.fp8, dn, slots * (L.H / 128), st);
  rec(5);
  return err;
}

}  // namespace exl3
