// Grouped GEMV path for decode-sized steps (a few tokens per expert).
//
// Page "GLM-5.3-Flash EXL3 (~2.1 bpw, SM70 tile order)", Running it: the
// expert kernels decode the trellis inside the matmul; Speed: direct per-lane
// window loads of strip-major tiles with deep prefetch.  Page "GLM-5.3 Flash
// EXL3 for 2x DGX Sparks", section Cold prefill (E3): gather, gate/up +
// SwiGLU, down + scatter, driven by device-side segment tables.
//
// Work item = (token group of <= 8 positions of one expert, projection,
// 128-output strip, K split).  A persistent grid walks the items.  Each of
// the 8 warps of a CTA takes every 8th 16-input block of the item and runs its
// own asynchronous-copy ring (cp.async, 16 bytes per lane, several blocks
// ahead, across item boundaries): per block the code row of the strip (8
// consecutive tiles, 8K bytes per lane) and the matching activation rows
// (8 tokens x 16 inputs).  Every lane then decodes its 64 weights in
// registers (the 16-K bit window overlap comes from the next lane of the quad
// by shuffle) and feeds mma.m16n8k16 with the K dimension doubled: the A
// register of weight (o, i) is the codebook's {a, b} fp16 pair itself and the
// B register holds {x_i, x_i}, so the tensor core forms (a + b) x_i with no
// separate add.  (The exact a + b differs from the format's fp16(a + b) by at
// most half an fp16 ulp; with the E4M3 rule the rounded value is formed first
// and placed as {v, 0}.)  Gate and up are separate items; SwiGLU runs in the
// down projection's input pass.
//
// Partial sums of the 8 warps are added in a fixed tree order in shared
// memory; K splits write their partials to the workspace and the CTA that
// completes an item last (atomic ticket) adds them in split order.  The
// result does not depend on scheduling and no atomics touch the data.
//
// Activations enter as fp16 with a power-of-two scale per (pair, projection)
// chosen from the row's max |x * suh| and undone in the epilogue, so the fp16
// operand never overflows whatever the input magnitude.
#include "common.cuh"
#include "internal.h"
#include "pipeline.cuh"

namespace exl3 {

namespace {

constexpr int kCW = 8;                     // warps per CTA
constexpr int kThreads = kCW * 32;
constexpr int kXsChunk = kGroup * 16 * 4;  // 8 tokens x 16 inputs x fp16x2

template <int K>
struct Cfg {
  static constexpr int kCodeChunk = 8 * 32 * K;  // 8 tiles of one 16-input block
  static constexpr int kSlot = kCodeChunk + kXsChunk;
  static constexpr int kStages = K == 2 ? 6 : (K == 3 ? 5 : 4);  // per-warp ring depth
  static constexpr int kWarpRing = kStages * kSlot;
  static constexpr int kRedOff = kCW * kWarpRing;
  static constexpr int kSmem = kRedOff + 4 * 1024 * 4;  // tree-reduction buffer
};

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

// Token group and slot of a segment position.
__device__ __forceinline__ void group_of(const int32_t* seg_offsets, const int32_t* group_off, int e,
                                         int pos, int* g, int* slot) {
  const int l = pos - seg_offsets[e];
  *g = group_off[e] + l / kGroup;
  *slot = l % kGroup;
}

// x rows of the pairs, times suh of gate and up, scaled, into the
// group-interleaved layout [group][proj][in/16][8 tokens][16] (fp16x2).
__global__ void __launch_bounds__(256) gather_xs_kernel(const void* __restrict__ x, int x_bf16,
                                                        int H, int k, RouteBuffers rb,
                                                        const uint16_t* __restrict__ suh_g,
                                                        const uint16_t* __restrict__ suh_u,
                                                        uint32_t* __restrict__ xs,
                                                        float* __restrict__ xs_inv) {
  __shared__ float s_tmp[32];
  const int pos = blockIdx.x;
  const int p = rb.seg_pairs[pos];
  const int t = p / k, e = rb.ids[p];
  int g, slot;
  group_of(rb.seg_offsets, rb.group_off, e, pos, &g, &slot);
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
  const int nb = H / 16;
  uint32_t* og = xs + (size_t)g * 2 * nb * kXsChunk / 4;
  uint32_t* ou = og + (size_t)nb * kXsChunk / 4;
  for (int idx = threadIdx.x; idx < H; idx += blockDim.x) {
    const float xv = load_act(x, x_bf16, (size_t)t * H + idx);
    const size_t dst = ((size_t)(idx >> 4) * kGroup + slot) * 16 + perm_slot(idx);
    og[dst] = dup_f16(xv * __half2float(__ushort_as_half(sg[idx])) * scg);
    ou[dst] = dup_f16(xv * __half2float(__ushort_as_half(su[idx])) * scu);
  }
  if (threadIdx.x == 0) {
    xs_inv[2 * pos] = ldexpf(1.0f, -eg);
    xs_inv[2 * pos + 1] = ldexpf(1.0f, -eu);
  }
}

// h = silu(g) * u for each position's row, times suh of down, scaled,
// group-interleaved (the down projection's B operand).
__global__ void __launch_bounds__(256) prep_down_kernel(const float* __restrict__ gu, size_t n_pos,
                                                        int I, RouteBuffers rb,
                                                        const uint16_t* __restrict__ suh_d,
                                                        uint32_t* __restrict__ xs,
                                                        float* __restrict__ xs_inv) {
  __shared__ float s_tmp[32];
  const int pos = blockIdx.x;
  const int e = rb.ids[rb.seg_pairs[pos]];
  int g, slot;
  group_of(rb.seg_offsets, rb.group_off, e, pos, &g, &slot);
  const uint16_t* sd = suh_d + (size_t)e * I;
  const float* gr = gu + (size_t)pos * I;
  const float* ur = gu + (n_pos + pos) * I;
  float am = 0.0f;
  for (int idx = threadIdx.x; idx < I; idx += blockDim.x)
    am = fmaxf(am, fabsf(silu_f(gr[idx]) * ur[idx] * __half2float(__ushort_as_half(sd[idx]))));
  am = block_max(am, s_tmp);
  const int ex = fp16_scale_exp(am);
  const float sc = ldexpf(1.0f, ex);
  uint32_t* o = xs + (size_t)g * (I / 16) * kXsChunk / 4;
  for (int idx = threadIdx.x; idx < I; idx += blockDim.x)
    o[((size_t)(idx >> 4) * kGroup + slot) * 16 + perm_slot(idx)] =
        dup_f16(silu_f(gr[idx]) * ur[idx] * __half2float(__ushort_as_half(sd[idx])) * sc);
  if (threadIdx.x == 0) xs_inv[pos] = ldexpf(1.0f, -ex);
}

template <int K, int FP8>
__device__ __forceinline__ void decode_mma(const LaneWords<K>& lw, const uint4& b,
                                           float (&acc)[8][4], uint32_t mult) {
  const uint32_t neg16 = opaque_u32(0xFFFF0000u);
#pragma unroll
  for (int r0 = 0; r0 < 8; r0++) {
#pragma unroll
    for (int hf = 0; hf < 2; hf++) {
      const int u = 8 * r0 + 4 * hf;
      uint32_t a0, a1, a2, a3;
      const uint32_t m0 = lane_halves<K>(lw, u + 0, mult, neg16);
      const uint32_t m1 = lane_halves<K>(lw, u + 1, mult, neg16);
      const uint32_t m2 = lane_halves<K>(lw, u + 2, mult, neg16);
      const uint32_t m3 = lane_halves<K>(lw, u + 3, mult, neg16);
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

template <int K>
__device__ __forceinline__ void lds_lane_words(LaneWords<K>& lw, const uint8_t* p) {
  if constexpr (K == 2) {
    const uint4 v = *reinterpret_cast<const uint4*>(p);
    lw.w[0] = v.x; lw.w[1] = v.y; lw.w[2] = v.z; lw.w[3] = v.w;
  } else if constexpr (K == 3) {
#pragma unroll
    for (int q = 0; q < 3; q++) {
      const uint2 v = *reinterpret_cast<const uint2*>(p + 8 * q);
      lw.w[2 * q] = v.x; lw.w[2 * q + 1] = v.y;
    }
  } else {
#pragma unroll
    for (int q = 0; q < 2; q++) {
      const uint4 v = *reinterpret_cast<const uint4*>(p + 16 * q);
      lw.w[4 * q] = v.x; lw.w[4 * q + 1] = v.y; lw.w[4 * q + 2] = v.z; lw.w[4 * q + 3] = v.w;
    }
  }
}

struct GemvParams {
  const uint16_t* codes[2];
  size_t stride[2];        // uint16 words per expert
  int in, out;
  int nproj;               // projections in this launch (2: gate and up)
  uint32_t mult;
  const uint16_t* svh[2];  // [E][out]
  const uint32_t* xs;      // [group][nproj][in/16][8][16] fp16x2
  const float* xs_inv;     // [pos][nproj]
  const int32_t* groups;   // [g][4] {expert, pos0, count, 0}
  const int32_t* n_groups; // device scalar
  const int32_t* seg_pairs;
  const float* wts;        // router weights by pair id (down launch)
  float* gu_out;           // gate/up launch: [proj][pos][out]
  float* r_out;            // down launch: [pair id][out]
  float* partial;          // [group][nproj][strip][nsplit][1024]
  int32_t* counters;       // [group][nproj][strip], zero on entry, left zero
  int32_t* status;
  int nsplit;
  size_t n_pos;            // positions (row count of gu_out per projection)
};

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <int K, int FP8>
__global__ void __launch_bounds__(kThreads, 3) gemv_kernel(GemvParams p) {
  using C = Cfg<K>;
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* ring = smem + warp * C::kWarpRing;
  float* red = reinterpret_cast<float*>(smem + C::kRedOff);
  const int strips = p.out / 128;
  const int nblk = p.in / 16;
  const int bps = nblk / p.nsplit;   // blocks per item
  const int bpw = bps / kCW;         // blocks per warp per item
  const int n_items = p.n_groups[0] * p.nproj * p.nsplit * strips;
  const int my_items = n_items > (int)blockIdx.x ? (n_items - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  const int n_jobs = my_items * bpw;  // this warp's blocks, across its items
  const size_t row_bytes = (size_t)(p.out / 16) * 32 * K;

  // item id -> (group, projection, split, strip); consecutive ids are
  // neighbouring strips, so concurrent CTAs read adjacent code bytes
  auto item_of = [&](int it, int& g, int& pj, int& q, int& s) {
    s = it % strips;
    int r = it / strips;
    q = r % p.nsplit;
    r /= p.nsplit;
    pj = r % p.nproj;
    g = r / p.nproj;
  };
  // copy the data of this warp's job j into ring slot j % kStages
  auto issue = [&](int j) {
    const int it = blockIdx.x + (j / bpw) * gridDim.x;
    int g, pj, q, s;
    item_of(it, g, pj, q, s);
    const int e = p.groups[4 * g];
    const int blk = q * bps + (j % bpw) * kCW + warp;
    uint8_t* slot = ring + (j % C::kStages) * C::kSlot;
    const uint8_t* cs = reinterpret_cast<const uint8_t*>(p.codes[pj] + p.stride[pj] * e) +
                        (size_t)blk * row_bytes + (size_t)8 * s * 32 * K;
#pragma unroll
    for (int c = 0; c < (C::kCodeChunk + 511) / 512; c++)
      if (c * 512 + lane * 16 < C::kCodeChunk) cp_async16(slot + c * 512 + lane * 16, cs + c * 512 + lane * 16);
    // activation rows: lane l copies 16 bytes of token slot l / 4; slots the
    // group does not fill are left alone (their MMA columns are discarded)
    if ((lane >> 2) < p.groups[4 * g + 2]) {
      const uint8_t* xsrc = reinterpret_cast<const uint8_t*>(p.xs) +
                            (((size_t)g * p.nproj + pj) * nblk + blk) * kXsChunk;
      cp_async16(slot + C::kCodeChunk + lane * 16, xsrc + lane * 16);
    }
  };

#pragma unroll
  for (int j = 0; j < C::kStages - 1; j++) {
    if (j < n_jobs) issue(j);
    cp_async_commit();
  }

  const int g_l = lane >> 2, c_l = lane & 3;
  int j = 0;
  for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
    int g, pj, q, s;
    item_of(item, g, pj, q, s);
    const int cnt = p.groups[4 * g + 2];
    float acc[8][4];
#pragma unroll
    for (int i = 0; i < 8; i++)
#pragma unroll
      for (int d = 0; d < 4; d++) acc[i][d] = 0.0f;
    for (int b = 0; b < bpw; b++, j++) {
      if (j + C::kStages - 1 < n_jobs) issue(j + C::kStages - 1);
      cp_async_commit();
      cp_async_wait<C::kStages - 1>();
      __syncwarp();
      const uint8_t* slot = ring + (j % C::kStages) * C::kSlot;
      LaneWords<K> lw;
      lds_lane_words<K>(lw, slot + lane * 8 * K);
      fetch_neighbour<K>(lw);
      const uint4 bx = g_l < cnt ? *reinterpret_cast<const uint4*>(slot + C::kCodeChunk + g_l * 64 + c_l * 16)
                                 : make_uint4(0, 0, 0, 0);
      decode_mma<K, FP8>(lw, bx, acc, p.mult);
      __syncwarp();  // the slot is refilled by the next iteration's issue
    }
    // fixed-order tree reduction over the 8 warps: 4+4, 2+2, 1+1
#pragma unroll
    for (int half = 4; half >= 1; half >>= 1) {
      if (warp >= half && warp < 2 * half) {
        float* dst = red + (size_t)(warp - half) * 1024;
#pragma unroll
        for (int i = 0; i < 8; i++)
          *reinterpret_cast<float4*>(dst + (i * 32 + lane) * 4) =
              make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
      }
      __syncthreads();
      if (warp < half) {
        const float* src = red + (size_t)warp * 1024;
#pragma unroll
        for (int i = 0; i < 8; i++) {
          const float4 v = *reinterpret_cast<const float4*>(src + (i * 32 + lane) * 4);
          acc[i][0] += v.x; acc[i][1] += v.y; acc[i][2] += v.z; acc[i][3] += v.w;
        }
      }
      __syncthreads();
    }
    if (warp == 0) {
      bool do_epi = true;
      if (p.nsplit > 1) {
        const size_t slot = ((size_t)g * p.nproj + pj) * strips + s;
        float* mine = p.partial + (slot * p.nsplit + q) * 1024;
#pragma unroll
        for (int i = 0; i < 8; i++)
          *reinterpret_cast<float4*>(mine + (i * 32 + lane) * 4) =
              make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
        __threadfence();
        __syncwarp();
        int last = 0;
        if (lane == 0) last = atomicAdd(&p.counters[slot], 1) == p.nsplit - 1;
        last = __shfl_sync(0xffffffffu, last, 0);
        do_epi = last;
        if (last) {
          __threadfence();
#pragma unroll
          for (int i = 0; i < 8; i++)
#pragma unroll
            for (int d = 0; d < 4; d++) acc[i][d] = 0.0f;
          for (int qq = 0; qq < p.nsplit; qq++) {
            const float* src = p.partial + (slot * p.nsplit + qq) * 1024;
#pragma unroll
            for (int i = 0; i < 8; i++) {
              const float4 v = __ldcg(reinterpret_cast<const float4*>(src + (i * 32 + lane) * 4));
              acc[i][0] += v.x; acc[i][1] += v.y; acc[i][2] += v.z; acc[i][3] += v.w;
            }
          }
          if (lane == 0) p.counters[slot] = 0;
        }
      }
      if (do_epi) {
        const int e = p.groups[4 * g], pos0 = p.groups[4 * g + 1], cnt = p.groups[4 * g + 2];
#pragma unroll
        for (int i = 0; i < 8; i++)
#pragma unroll
          for (int d = 0; d < 4; d++) {
            const int o = 16 * (8 * s + g_l) + i + 8 * (d >> 1);
            const int n = 2 * c_l + (d & 1);
            if (n < cnt) {
              const int pos = pos0 + n;
              const float v = acc[i][d] * p.xs_inv[(size_t)pos * p.nproj + pj] *
                              __half2float(__ushort_as_half(p.svh[pj][(size_t)e * p.out + o]));
              if (p.gu_out) {
                p.gu_out[((size_t)pj * p.n_pos + pos) * p.out + o] = v;
              } else {
                const int pid = p.seg_pairs[pos];
                p.r_out[(size_t)pid * p.out + o] = v * p.wts[pid];
              }
            }
          }
      }
    }
  }
  cp_async_wait<0>();
}

template <int K, int FP8>
cudaError_t launch_gemv(const GemvParams& gp, int items_ub, cudaStream_t st) {
  using C = Cfg<K>;
  static int occ = -1, sms = 0;
  auto kfn = gemv_kernel<K, FP8>;
  if (occ < 0) {
    cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kfn, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int o = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, kfn, kThreads, C::kSmem);
    occ = o < 1 ? 1 : o;
  }
  int grid = sms * occ;
  if (items_ub < grid) grid = items_ub;
  if (grid < 1) grid = 1;
  kfn<<<grid, kThreads, C::kSmem, st>>>(gp);
  note_launches(1);
  return cudaGetLastError();
}

cudaError_t dispatch_gemv(int K, int fp8, const GemvParams& gp, int items_ub, cudaStream_t st) {
  if (fp8) {
    if (K == 2) return launch_gemv<2, 1>(gp, items_ub, st);
    if (K == 3) return launch_gemv<3, 1>(gp, items_ub, st);
    return launch_gemv<4, 1>(gp, items_ub, st);
  }
  if (K == 2) return launch_gemv<2, 0>(gp, items_ub, st);
  if (K == 3) return launch_gemv<3, 0>(gp, items_ub, st);
  return launch_gemv<4, 0>(gp, items_ub, st);
}

// K splits: double while every warp keeps >= 2 blocks per item and the upper
// bound on items stays below ~6 per CTA slot (3 CTAs on 152 SMs).
int choose_nsplit(size_t groups_ub, int items_per_group, int nblk) {
  int ns = 1;
  while (ns < 8 && nblk % (2 * ns * kCW) == 0 && nblk / (2 * ns * kCW) >= 2 &&
         groups_ub * items_per_group * ns < (size_t)6 * 456)
    ns *= 2;
  return ns;
}

size_t al(size_t b) { return (b + 255) & ~(size_t)255; }

struct GemvLayout {
  size_t xs_gu, xs_gu_inv, gu, xs_d, xs_d_inv, r, partial, counters, total;
  int ns_gu, ns_d;
  size_t n_counters;
};

GemvLayout gemv_layout(int T, int top_k, int E, int H, int I) {
  GemvLayout g{};
  const size_t P = (size_t)T * top_k;
  const size_t G = max_groups(T, E, top_k);
  g.ns_gu = choose_nsplit(G, 2 * (I / 128), H / 16);
  g.ns_d = choose_nsplit(G, H / 128, I / 16);
  const size_t part_gu = g.ns_gu > 1 ? G * 2 * (I / 128) * g.ns_gu * 1024 * 4 : 0;
  const size_t part_d = g.ns_d > 1 ? G * (H / 128) * g.ns_d * 1024 * 4 : 0;
  g.n_counters = G * (2 * (I / 128) > H / 128 ? 2 * (I / 128) : H / 128);
  size_t o = 0;
  g.xs_gu = o; o += al(G * 2 * (H / 16) * kXsChunk);
  g.xs_gu_inv = o; o += al(P * 2 * 4);
  g.gu = o; o += al(2 * P * I * 4);
  g.xs_d = o; o += al(G * (I / 16) * kXsChunk);
  g.xs_d_inv = o; o += al(P * 4);
  g.r = o; o += al(P * H * 4);
  g.partial = o; o += al(part_gu > part_d ? part_gu : part_d);
  g.counters = o; o += al(g.n_counters * 4);
  g.total = o;
  return g;
}

}  // namespace

size_t gemv_scratch_bytes(int T, int top_k, int E, int H, int I) {
  return gemv_layout(T, top_k, E, H, I).total;
}

void gemv_carve(void* ws, int T, int top_k, int E, int H, int I, GemvBuffers* gb) {
  const GemvLayout g = gemv_layout(T, top_k, E, H, I);
  char* q = static_cast<char*>(ws);
  gb->xs_gu = reinterpret_cast<uint32_t*>(q + g.xs_gu);
  gb->xs_gu_inv = reinterpret_cast<float*>(q + g.xs_gu_inv);
  gb->gu = reinterpret_cast<float*>(q + g.gu);
  gb->xs_d = reinterpret_cast<uint32_t*>(q + g.xs_d);
  gb->xs_d_inv = reinterpret_cast<float*>(q + g.xs_d_inv);
  gb->r = reinterpret_cast<float*>(q + g.r);
  gb->partial = reinterpret_cast<float*>(q + g.partial);
  gb->counters = reinterpret_cast<int32_t*>(q + g.counters);
  gb->n_counters = g.n_counters;
  gb->ns_gu = g.ns_gu;
  gb->ns_d = g.ns_d;
}

cudaError_t launch_moe_gemv(const LayerView& L, const void* x, int x_bf16, int T, int top_k,
                            const RouteBuffers& rb, const GemvBuffers& gb, const cudaEvent_t* ev,
                            cudaStream_t st) {
  auto rec = [&](int i) {
    if (ev && ev[i]) record_stage_event(ev[i], st);
  };
  const int P = T * top_k;
  const size_t G = max_groups(T, L.E, top_k);
  cudaError_t err;
  if ((err = cudaMemsetAsync(gb.counters, 0, gb.n_counters * sizeof(int32_t), st)) != cudaSuccess)
    return err;
  gather_xs_kernel<<<P, 256, 0, st>>>(x, x_bf16, L.H, top_k, rb, L.suh[0], L.suh[1], gb.xs_gu,
                                      gb.xs_gu_inv);
  note_launches(1);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  rec(2);

  // gate and up share one launch, so they share a width (checked at create)
  GemvParams gu{};
  gu.codes[0] = L.codes[0]; gu.codes[1] = L.codes[1];
  gu.stride[0] = L.code_stride[0]; gu.stride[1] = L.code_stride[1];
  gu.in = L.H; gu.out = L.I; gu.nproj = 2; gu.mult = L.mult;
  gu.svh[0] = L.svh[0]; gu.svh[1] = L.svh[1];
  gu.xs = gb.xs_gu; gu.xs_inv = gb.xs_gu_inv;
  gu.groups = rb.groups; gu.n_groups = rb.group_off + L.E;
  gu.seg_pairs = rb.seg_pairs; gu.wts = rb.w; gu.gu_out = gb.gu; gu.n_pos = (size_t)P;
  gu.partial = gb.partial; gu.counters = gb.counters; gu.status = rb.status;
  gu.nsplit = gb.ns_gu;
  if ((err = dispatch_gemv(L.K[0], L.fp8, gu, (int)(G * 2 * (L.I / 128) * gu.nsplit), st)) !=
      cudaSuccess)
    return err;
  rec(3);

  prep_down_kernel<<<P, 256, 0, st>>>(gb.gu, (size_t)P, L.I, rb, L.suh[2], gb.xs_d, gb.xs_d_inv);
  note_launches(1);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  rec(4);

  GemvParams dn{};
  dn.codes[0] = L.codes[2]; dn.stride[0] = L.code_stride[2];
  dn.in = L.I; dn.out = L.H; dn.nproj = 1; dn.mult = L.mult;
  dn.svh[0] = L.svh[2];
  dn.xs = gb.xs_d; dn.xs_inv = gb.xs_d_inv;
  dn.groups = rb.groups; dn.n_groups = rb.group_off + L.E;
  dn.seg_pairs = rb.seg_pairs; dn.wts = rb.w; dn.r_out = gb.r;
  dn.partial = gb.partial; dn.counters = gb.counters; dn.status = rb.status;
  dn.nsplit = gb.ns_d;
  err = dispatch_gemv(L.K[2], L.fp8, dn, (int)(G * (L.H / 128) * dn.nsplit), st);
  rec(5);
  return err;
}

}  // namespace exl3
