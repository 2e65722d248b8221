// Grouped GEMV path for decode-sized steps (a few tokens per expert).
//
// Page "GLM-5.3-Flash EXL3 (~2.1 bpw, SM70 tile order)", Running it: the
// expert kernels decode the trellis inside the matmul; Speed: direct per-lane
// window loads of strip-major tiles with deep prefetch.  Page "GLM-5.3 Flash
// EXL3 for 2x DGX Sparks", section Cold prefill (E3): gather, gate/up +
// SwiGLU, down + scatter, driven by device-side segment tables.
//
// Work item = (token group of <= 8 positions of one expert, projection,
// 128-output strip, K split), processed by ONE warp; warps take items from a
// device counter (an item's successor is taken while its last blocks are
// still being copied), so the load stays balanced whatever the expert mix.
// Each warp runs its own asynchronous-copy ring (cp.async, 16 bytes per lane,
// several jobs of two 16-input blocks ahead, across item boundaries): per
// block the code row of the strip (8 consecutive tiles, 8K bytes per lane) and
// the matching activation rows (8 tokens x 16 inputs).  Every lane then decodes its 64
// weights in registers (the 16-K bit window overlap comes from the next lane
// of the quad by shuffle) and feeds mma.m16n8k16 with the K dimension
// doubled: the A register of weight (o, i) is the codebook's {a, b} fp16 pair
// itself and the B register holds {x_i, x_i}, so the tensor core forms
// (a + b) x_i with no separate add.  (The exact a + b differs from the
// format's fp16(a + b) by at most half an fp16 ulp; with the E4M3 rule the
// rounded value is formed first and placed as {v, 0}.)  Gate and up are
// separate items; SwiGLU runs in the down projection's input pass.
//
// Every item writes its scaled partial sums to its own K-split slab; the
// consumers (the down projection's input pass, the combine) add the slabs in
// split order, so the result does not depend on scheduling and no atomics
// touch the data.
//
// Activations enter as fp16 with a power-of-two scale per (pair, projection)
// chosen from the row's max |x * suh| and undone in the epilogue, so the fp16
// operand never overflows whatever the input magnitude.
//
// Format v2 (Hadamard rotation): the input passes rotate each 128-input block
// of x * suh (h * suh for down) before the scale is chosen: a thread's 16
// inputs in registers, the 8 threads of a block by shuffles.  The epilogue
// rotates each item's partial sums over its 128-output strip (16 outputs of a
// lane in registers, the 8 lane quads by shuffles) before svh; the rotation
// is linear, so rotating every K-split partial equals rotating their sum.
#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "pipeline.cuh"

namespace exl3 {

namespace {

constexpr int kCW = 8;                     // warps per CTA
constexpr int kThreads = kCW * 32;
constexpr int kXsChunk = kGroup * 16 * 4;  // 8 tokens x 16 inputs x fp16x2
constexpr int kJobBlocks = 2;              // 16-input blocks per ring job

template <int K>
struct Cfg {
  static constexpr int kCodeChunk = 8 * 32 * K;  // 8 tiles of one 16-input block
  static constexpr int kBlkBytes = kCodeChunk + kXsChunk;
  static constexpr int kSlot = kJobBlocks * kBlkBytes;              // one job: 2 blocks
  // per-warp ring depth in jobs; at most 4, the fewest jobs of an item
  // (8 blocks), which keeps the producer within one item of the consumer
  static constexpr int kStages = K == 4 ? 3 : 4;
  static constexpr int kWarpRing = kStages * kSlot;
  static constexpr int kSmem = kCW * kWarpRing;
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

// Activation slots inside a 16-input block: lane c of an MMA quad reads
// slots 4c..4c+3, which hold inputs c, c+4, c+8, c+12 (slot q holds input
// 4 (q & 3) + (q >> 2)).

// Token group and slot of a segment position.
__device__ __forceinline__ void group_of(const int32_t* seg_offsets, const int32_t* group_off, int e,
                                         int pos, int* g, int* slot) {
  const int l = pos - seg_offsets[e];
  *g = group_off[e] + l / kGroup;
  *slot = l % kGroup;
}

// Both input passes below (launched with input_pass_threads: whole warps,
// blockDim a multiple of 8) give each thread one 16-input block per step
// (16-byte loads of x / suh, float4 loads of fp32 rows), keep its first block
// in registers between the max pass and the write pass (re-reading any
// further ones), and write the block's 16 token-slot values as four 16-byte
// stores in the permuted slot order; one CTA per position.
__device__ __forceinline__ void f16x8(const uint4& r, float* f, int bf16) {
  const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
  for (int i = 0; i < 4; i++) {
    const uint32_t lo = w[i] & 0xFFFFu, hi = w[i] >> 16;
    if (bf16) {
      f[2 * i] = __uint_as_float(lo << 16);
      f[2 * i + 1] = __uint_as_float(hi << 16);
    } else {
      f[2 * i] = __half2float(__ushort_as_half((unsigned short)lo));
      f[2 * i + 1] = __half2float(__ushort_as_half((unsigned short)hi));
    }
  }
}

// Store the 16 inputs of block b of one token slot into the group-interleaved
// layout, each value duplicated into fp16x2, in the slot order above.
__device__ __forceinline__ void put16(uint32_t* o, int b, int slot, const float (&f)[16], float sc) {
  uint4* d = reinterpret_cast<uint4*>(o + ((size_t)b * kGroup + slot) * 16);
#pragma unroll
  for (int v = 0; v < 4; v++) {
    uint32_t w[4];
#pragma unroll
    for (int u = 0; u < 4; u++) {
      const int q = 4 * v + u;
      w[u] = dup_f16(f[4 * (q & 3) + (q >> 2)] * sc);
    }
    d[v] = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// Format v2: rotate the 128-input block of which this thread holds 16
// consecutive inputs (threads 8j .. 8j+7 hold one block, all active).
__device__ __forceinline__ void rotate_block16(float (&f)[16]) {
  wht_regs(f);
  const unsigned gm = 0xFFu << (threadIdx.x & 24);
#pragma unroll
  for (int m = 1; m < 8; m <<= 1)
#pragma unroll
    for (int q = 0; q < 16; q++) f[q] = wht_lane(f[q], m, gm);
}

// FP8 operand mode: the 16 values as their E4M3 operand values q = E4M3(a / s)
// (exact in fp16, so the GEMV's fp16 operand carries them unchanged).
__device__ __forceinline__ void quant16(float (&f)[16], float s) {
  const float r = s > 0.0f ? __frcp_rn(s) : 0.0f;
#pragma unroll
  for (int q = 0; q < 16; q++) f[q] = e4m3_value(f[q], s, r);
}

__device__ __forceinline__ float amax16(float a, const float (&f)[16]) {
#pragma unroll
  for (int q = 0; q < 16; q++) a = fmaxf(a, fabsf(f[q]));
  return a;
}

// x rows of the pairs, times suh of gate and up (rotated when had), scaled,
// into the group-interleaved layout [group][proj][in/16][8 tokens][16]
// (fp16x2).  blockDim is a multiple of 8, so thread b's block shares its
// 128-input block with threads b ^ 1 .. b ^ 7 in every step.  act8 (FP8
// operand mode): the rows' E4M3 operand values with their fp32 row scales
// instead of a power-of-two scale.
__global__ void __launch_bounds__(256) gather_xs_kernel(const void* __restrict__ x, int x_bf16,
                                                        int H, int k, RouteBuffers rb,
                                                        const uint16_t* __restrict__ suh_g,
                                                        const uint16_t* __restrict__ suh_u,
                                                        int had, int act8, Shard sh,
                                                        uint32_t* __restrict__ xs,
                                                        float* __restrict__ xs_inv,
                                                        int32_t* __restrict__ zero_ctrs) {
  pdl_wait();
  // the work counters of the GEMV launches that follow start at zero; null
  // when a memset has already cleared them
  if (zero_ctrs && blockIdx.x == 0 && threadIdx.x < 12) zero_ctrs[threadIdx.x] = 0;
  __shared__ float s_tmp[32];
  const int pos = blockIdx.x;
  const int p = rb.seg_pairs[pos];
  const int t = p / k, e = rb.ids[p];
  if (e < sh.e0 || e >= sh.e1) return;  // another call's expert (whole CTA)
  int g, slot;
  group_of(rb.seg_offsets, rb.group_off, e, pos, &g, &slot);
  const uint4* xv = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(x) + (size_t)t * H);
  const uint4* sg = reinterpret_cast<const uint4*>(suh_g + (size_t)e * H);
  const uint4* su = reinterpret_cast<const uint4*>(suh_u + (size_t)e * H);
  const int nb = H / 16;
  // products x * suh of block b
  auto prod = [&](int b, float (&fg)[16], float (&fu)[16]) {
    float fx[16], a[16], c[16];
    f16x8(xv[2 * b], fx, x_bf16);
    f16x8(xv[2 * b + 1], fx + 8, x_bf16);
    f16x8(sg[2 * b], a, 0);
    f16x8(sg[2 * b + 1], a + 8, 0);
    f16x8(su[2 * b], c, 0);
    f16x8(su[2 * b + 1], c + 8, 0);
#pragma unroll
    for (int q = 0; q < 16; q++) {
      fg[q] = fx[q] * a[q];
      fu[q] = fx[q] * c[q];
    }
    if (had) {
      rotate_block16(fg);
      rotate_block16(fu);
    }
  };
  float cg[16], cu[16];
  float ag = 0.0f, au = 0.0f;
  const int b0 = threadIdx.x;
  if (b0 < nb) {
    prod(b0, cg, cu);
    ag = amax16(ag, cg);
    au = amax16(au, cu);
  }
  for (int b = b0 + blockDim.x; b < nb; b += blockDim.x) {
    float fg[16], fu[16];
    prod(b, fg, fu);
    ag = amax16(ag, fg);
    au = amax16(au, fu);
  }
  ag = block_max(ag, s_tmp);
  au = block_max(au, s_tmp);
  const int eg = fp16_scale_exp(ag), eu = fp16_scale_exp(au);
  const float qg = e4m3_row_scale(ag), qu = e4m3_row_scale(au);
  const float scg = act8 ? 1.0f : ldexpf(1.0f, eg), scu = act8 ? 1.0f : ldexpf(1.0f, eu);
  uint32_t* og = xs + (size_t)g * 2 * nb * kXsChunk / 4;
  uint32_t* ou = og + (size_t)nb * kXsChunk / 4;
  auto put2 = [&](int b, float (&fg)[16], float (&fu)[16]) {
    if (act8) {
      quant16(fg, qg);
      quant16(fu, qu);
    }
    put16(og, b, slot, fg, scg);
    put16(ou, b, slot, fu, scu);
  };
  if (b0 < nb) put2(b0, cg, cu);
  for (int b = b0 + blockDim.x; b < nb; b += blockDim.x) {
    float fg[16], fu[16];
    prod(b, fg, fu);
    put2(b, fg, fu);
  }
  if (threadIdx.x == 0) {
    const int hs = had ? kHadShift : 0;  // the unnormalized rotations' 128
    xs_inv[2 * pos] = act8 ? ldexpf(qg, -hs) : ldexpf(1.0f, -eg - hs);
    xs_inv[2 * pos + 1] = act8 ? ldexpf(qu, -hs) : ldexpf(1.0f, -eu - hs);
  }
}

// h = silu(g) * u for each position's row (g and u summed over the gate/up
// launch's K splits in split order), times suh of down (rotated when had),
// scaled, group-interleaved (the down projection's B operand).
__global__ void __launch_bounds__(256) prep_down_kernel(const float* __restrict__ gu, int ns,
                                                        size_t n_pos, int I, RouteBuffers rb,
                                                        const uint16_t* __restrict__ suh_d,
                                                        int had, int act8, Shard sh,
                                                        uint32_t* __restrict__ xs,
                                                        float* __restrict__ xs_inv) {
  pdl_wait();
  __shared__ float s_tmp[32];
  const int pos = blockIdx.x;
  const int e = rb.ids[rb.seg_pairs[pos]];
  if (e < sh.e0 || e >= sh.e1) return;  // another call's expert (whole CTA)
  int g, slot;
  group_of(rb.seg_offsets, rb.group_off, e, pos, &g, &slot);
  const uint4* sd = reinterpret_cast<const uint4*>(suh_d + (size_t)e * I);
  // gate / up of split q: gu + ((q * 2 + proj) * n_pos + pos) * I
  const float4* gr = reinterpret_cast<const float4*>(gu + (size_t)pos * I);
  const float4* ur = reinterpret_cast<const float4*>(gu + (n_pos + pos) * I);
  const size_t qstride = 2 * n_pos * I / 4;  // float4s per split slab
  const int nb = I / 16;
  auto hval = [&](int b, float (&h)[16]) {
    float sv[16];
    f16x8(sd[2 * b], sv, 0);
    f16x8(sd[2 * b + 1], sv + 8, 0);
    float gg[16], uu[16];
#pragma unroll
    for (int q = 0; q < 16; q++) gg[q] = uu[q] = 0.0f;
#pragma unroll 2
    for (int q = 0; q < ns; q++) {  // K splits in order
#pragma unroll
      for (int c = 0; c < 4; c++) {
        const float4 a = __ldcs(gr + q * qstride + 4 * b + c);
        const float4 u = __ldcs(ur + q * qstride + 4 * b + c);
        gg[4 * c] += a.x; gg[4 * c + 1] += a.y; gg[4 * c + 2] += a.z; gg[4 * c + 3] += a.w;
        uu[4 * c] += u.x; uu[4 * c + 1] += u.y; uu[4 * c + 2] += u.z; uu[4 * c + 3] += u.w;
      }
    }
#pragma unroll
    for (int q = 0; q < 16; q++) h[q] = silu_f(gg[q]) * uu[q] * sv[q];
    if (had) rotate_block16(h);
  };
  float c[16];
  float am = 0.0f;
  const int b0 = threadIdx.x;
  if (b0 < nb) {
    hval(b0, c);
    am = amax16(am, c);
  }
  for (int b = b0 + blockDim.x; b < nb; b += blockDim.x) {
    float h[16];
    hval(b, h);
    am = amax16(am, h);
  }
  am = block_max(am, s_tmp);
  const int ex = fp16_scale_exp(am);
  const float qs = e4m3_row_scale(am);
  const float sc = act8 ? 1.0f : ldexpf(1.0f, ex);
  uint32_t* o = xs + (size_t)g * nb * kXsChunk / 4;
  if (b0 < nb) {
    if (act8) quant16(c, qs);
    put16(o, b0, slot, c, sc);
  }
  for (int b = b0 + blockDim.x; b < nb; b += blockDim.x) {
    float h[16];
    hval(b, h);
    if (act8) quant16(h, qs);
    put16(o, b, slot, h, sc);
  }
  if (threadIdx.x == 0)
    xs_inv[pos] = act8 ? ldexpf(qs, -(had ? kHadShift : 0)) : ldexpf(1.0f, -ex - (had ? kHadShift : 0));
}

template <int K, int FP8>
__device__ __forceinline__ void decode_mma(const LaneWords<K>& lw, const uint4& b,
                                           float (&acc)[8][4], uint32_t mult) {
  const uint32_t neg16 = opaque_u32(0xFFFF0000u);
  const McgConsts mc = mcg_consts();
  constexpr int step = K == 3 ? 0 : 16 / K;
  uint32_t xp[8 + (K == 3 ? 0 : 16 / K)];
  if constexpr (K != 3) {
#pragma unroll
    for (int t = 0; t < step; t++) xp[t] = lane_window32<K>(lw, t * K) * mult;
  }
#pragma unroll
  for (int r0 = 0; r0 < 8; r0++) {
    uint32_t m[8];
    if constexpr (K == 3) {
#pragma unroll
      for (int t = 0; t < 8; t++) m[t] = mcg_halves(lane_state<K>(lw, 8 * r0 + t), mult, mc);
    } else {
      // xp[0..step) already hold weights 8 r0 .. 8 r0 + step - 1
#pragma unroll
      for (int t = step; t < 8 + step; t++) xp[t] = lane_window32<K>(lw, (8 * r0 + t) * K) * mult;
#pragma unroll
      for (int t = 0; t < 8; t++) m[t] = mcg_maskxor(xp[t + step] * neg16 + xp[t], mc);
#pragma unroll
      for (int t = 0; t < step; t++) xp[t] = xp[t + 8];
    }
#pragma unroll
    for (int hf = 0; hf < 2; hf++) {
      uint32_t a0, a1, a2, a3;
      const uint32_t* mm = m + 4 * hf;
      if (!FP8) {
        a0 = mm[0]; a1 = mm[1]; a2 = mm[2]; a3 = mm[3];
      } else {
        const uint32_t v01 = e4m3_round2(sum_halves2(mm[0], mm[1]));
        const uint32_t v23 = e4m3_round2(sum_halves2(mm[2], mm[3]));
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
  const int32_t* g_begin;  // device scalar: first group of the call's expert range
  const int32_t* n_groups; // device scalar: end of the range's groups
  const int32_t* seg_pairs;
  const float* wts;        // router weights by pair id (down launch)
  float* gu_out;           // gate/up launch: [split][proj][pos][out]
  float* r_out;            // down launch: [split][pair id][out]
  size_t n_pos;            // positions = pairs
  int32_t* work;           // item counter, zero on entry
  int nsplit;
  // mixed widths: this launch's work list of (group, projection) pairs whose
  // width is this instantiation's K, and the experts' code offsets
  const int32_t* entries;  // [n][2], or null: every group, every projection
  const int32_t* n_entries;
  const unsigned long long* off;  // [E][3] code word offsets, or null: stride * e
  int proj0;               // global index of this launch's projection 0 (0 or 2)
};

// Mixed widths: split the token groups' (group, projection) work into one
// list per width.  Thread per (group, projection p of 3): gate and up go to
// the gate/up launch's lists, down to the down launch's.  The order inside a
// list does not matter (every item writes its own rows).
__global__ void __launch_bounds__(256) width_lists_kernel(const int32_t* __restrict__ n_groups,
                                                          const int32_t* __restrict__ groups,
                                                          const int32_t* __restrict__ kt,
                                                          int cap_gu, int cap_d, Shard sh,
                                                          int32_t* __restrict__ counts,
                                                          int32_t* __restrict__ entries) {
  pdl_wait();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= 3 * n_groups[0]) return;
  const int g = i / 3, pg = i % 3;
  if (groups[4 * g] < sh.e0 || groups[4 * g] >= sh.e1) return;  // another call's expert
  const int w = kt[(size_t)groups[4 * g] * 3 + pg] - 2;
  const int launch = pg == 2 ? 1 : 0;
  const int cap = launch ? cap_d : cap_gu;
  const int slot = atomicAdd(&counts[launch * 3 + w], 1);
  int32_t* e = entries + ((size_t)launch * 3 * cap_gu + (size_t)w * cap + slot) * 2;
  e[0] = g;
  e[1] = launch ? 0 : pg;
}

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Next item of the launch for this warp (warp-uniform).
__device__ __forceinline__ int grab_item(int32_t* work) {
  int it = 0;
  if ((threadIdx.x & 31) == 0) it = atomicAdd(work, 1);
  return __shfl_sync(0xffffffffu, it, 0);
}

template <int K, int FP8, int HAD>
__global__ void __launch_bounds__(kThreads, 2) gemv_kernel(GemvParams p) {
  using C = Cfg<K>;
  extern __shared__ __align__(128) uint8_t smem[];
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* ring = smem + warp * C::kWarpRing;
  const int strips = p.out / 128;
  const int nblk = p.in / 16;
  const int bps = nblk / p.nsplit;   // blocks (jobs) per item, >= kStages - 1
  const int g_first = p.g_begin[0];
  const int n_items =
      (p.entries ? p.n_entries[0] : (p.n_groups[0] - g_first) * p.nproj) * p.nsplit * strips;
  const size_t row_bytes = (size_t)(p.out / 16) * 32 * K;

  // item id -> (group, projection, split, strip); consecutive ids are
  // neighbouring strips, so warps taking consecutive items read adjacent code
  auto item_of = [&](int it, int& g, int& pj, int& q, int& s) {
    s = it % strips;
    int r = it / strips;
    q = r % p.nsplit;
    r /= p.nsplit;
    if (p.entries) {
      g = p.entries[2 * r];
      pj = p.entries[2 * r + 1];
    } else {
      pj = r % p.nproj;
      g = g_first + r / p.nproj;
    }
  };
  // first code word of projection pj of expert e
  auto expert_codes = [&](int e, int pj) {
    return (pj ? p.codes[1] : p.codes[0]) +
           (p.off ? (size_t)p.off[(size_t)e * 3 + p.proj0 + pj]
                  : (pj ? p.stride[1] : p.stride[0]) * (size_t)e);
  };
  // Producer cursor: the source addresses of the next block to copy.
  struct Cursor {
    int b;                  // block of the item (0..bps-1)
    const uint8_t* cs;      // code chunk of the block
    const uint8_t* xsrc;    // this lane's activation piece (nullptr: token slot unused)
  } cur;
  auto cursor_item = [&](int it) {
    int g, pj, q, s;
    item_of(it, g, pj, q, s);
    const int e = p.groups[4 * g];
    const int blk = q * bps;
    cur.b = 0;
    cur.cs = reinterpret_cast<const uint8_t*>(expert_codes(e, pj)) + (size_t)blk * row_bytes +
             (size_t)8 * s * 32 * K;
    // lane l copies 16 bytes of token slot l / 4; slots the group does not
    // fill are left alone (their MMA columns are discarded)
    cur.xsrc = (lane >> 2) < p.groups[4 * g + 2]
                   ? reinterpret_cast<const uint8_t*>(p.xs) +
                         (((size_t)g * p.nproj + pj) * nblk + blk) * kXsChunk + lane * 16
                   : nullptr;
  };

  int item = grab_item(p.work);
  if (item >= n_items) return;
  cursor_item(item);
  int next_item = n_items;  // taken by the producer when it leaves `item`
  bool p_done = false;
  // copy the cursor's next job (two blocks) into ring slot `slot_idx` and
  // advance the cursor.  The producer runs kStages - 1 jobs ahead of the
  // consumer; since an item has at least kStages jobs (bps >= 8 blocks), it
  // finishes issuing the next item only after the consumer has left the
  // current one, so next_item is never overwritten too early
  auto issue = [&](int slot_idx) {
    uint8_t* slot = ring + slot_idx * C::kSlot;
#pragma unroll
    for (int q = 0; q < kJobBlocks; q++) {
      uint8_t* dst = slot + q * C::kBlkBytes;
      const uint8_t* cs = cur.cs + q * row_bytes;
#pragma unroll
      for (int c = 0; c < (C::kCodeChunk + 511) / 512; c++)
        if (c * 512 + lane * 16 < C::kCodeChunk) cp_async16(dst + c * 512 + lane * 16, cs + c * 512 + lane * 16);
      if (cur.xsrc) cp_async16(dst + C::kCodeChunk + lane * 16, cur.xsrc + q * kXsChunk);
    }
    if ((cur.b += kJobBlocks) < bps) {
      cur.cs += kJobBlocks * row_bytes;
      if (cur.xsrc) cur.xsrc += kJobBlocks * kXsChunk;
    } else {
      next_item = grab_item(p.work);
      if (next_item < n_items) cursor_item(next_item);
      else p_done = true;
    }
  };

  int issue_slot = 0;
#pragma unroll
  for (int j = 0; j < C::kStages - 1; j++) {
    if (!p_done) issue(issue_slot);
    issue_slot = issue_slot + 1 == C::kStages ? 0 : issue_slot + 1;
    cp_async_commit();
  }
  int read_slot = 0;

  const int g_l = lane >> 2, c_l = lane & 3;
  while (item < n_items) {
    int g, pj, q, s;
    item_of(item, g, pj, q, s);
    const int e = p.groups[4 * g], pos0 = p.groups[4 * g + 1], cnt = p.groups[4 * g + 2];
    // epilogue scalars, loaded now so their latency hides behind the blocks:
    // this lane's 16 outputs (two runs of 8 svh values) and 2 token slots
    const int obase = 16 * (8 * s + g_l);
    const uint16_t* svh = (pj ? p.svh[1] : p.svh[0]) + (size_t)e * p.out + obase;
    const uint4 sv_lo = __ldg(reinterpret_cast<const uint4*>(svh));
    const uint4 sv_hi = __ldg(reinterpret_cast<const uint4*>(svh + 8));
    float tok_scale[2];
    int tok_row[2];
#pragma unroll
    for (int u = 0; u < 2; u++) {
      const int n = 2 * c_l + u;
      tok_scale[u] = 0.0f;
      tok_row[u] = 0;
      if (n < cnt) {
        const int pos = pos0 + n;
        tok_scale[u] = __ldg(p.xs_inv + (size_t)pos * p.nproj + pj);
        if (p.gu_out) {
          tok_row[u] = ((q * p.nproj + pj) * (int)p.n_pos + pos);
        } else {
          const int pid = __ldg(p.seg_pairs + pos);
          tok_scale[u] *= __ldg(p.wts + pid);
          tok_row[u] = q * (int)p.n_pos + pid;
        }
      }
    }
    float acc[8][4];
#pragma unroll
    for (int i = 0; i < 8; i++)
#pragma unroll
      for (int d = 0; d < 4; d++) acc[i][d] = 0.0f;
    for (int b = 0; b < bps; b += kJobBlocks) {
      if (!p_done) issue(issue_slot);
      issue_slot = issue_slot + 1 == C::kStages ? 0 : issue_slot + 1;
      cp_async_commit();
      cp_async_wait<C::kStages - 1>();
      __syncwarp();
      const uint8_t* slot = ring + read_slot * C::kSlot;
      read_slot = read_slot + 1 == C::kStages ? 0 : read_slot + 1;
#pragma unroll
      for (int q = 0; q < kJobBlocks; q++) {
        const uint8_t* blk = slot + q * C::kBlkBytes;
        LaneWords<K> lw;
        lds_lane_words<K>(lw, blk + lane * 8 * K);
        fetch_neighbour<K>(lw);
        const uint4 bx = g_l < cnt ? *reinterpret_cast<const uint4*>(blk + C::kCodeChunk + g_l * 64 + c_l * 16)
                                   : make_uint4(0, 0, 0, 0);
        decode_mma<K, FP8>(lw, bx, acc, p.mult);
      }
      __syncwarp();  // the slot is refilled by a later issue
    }
    if constexpr (HAD != 0) {
      // rotate over the strip's 128 outputs: lane (g_l, c_l) holds outputs
      // 16 g_l + 8 dh + i as acc[i][2 dh + u] for its tokens u = 0, 1
#pragma unroll
      for (int u = 0; u < 2; u++) {
        float v[16];
#pragma unroll
        for (int i = 0; i < 16; i++) v[i] = acc[i & 7][2 * (i >> 3) + u];
        wht_regs(v);
#pragma unroll
        for (int m = 4; m < 32; m <<= 1)
#pragma unroll
          for (int i = 0; i < 16; i++) v[i] = wht_lane(v[i], m, 0xffffffffu);
#pragma unroll
        for (int i = 0; i < 16; i++) acc[i & 7][2 * (i >> 3) + u] = v[i];
      }
    }
    // this item's scaled partial sums into its split slab
    float* dst = p.gu_out ? p.gu_out : p.r_out;
    const uint32_t svw[8] = {sv_lo.x, sv_lo.y, sv_lo.z, sv_lo.w, sv_hi.x, sv_hi.y, sv_hi.z, sv_hi.w};
#pragma unroll
    for (int i = 0; i < 8; i++)
#pragma unroll
      for (int d = 0; d < 4; d++) {
        const int u = d & 1, dh = d >> 1;
        if (2 * c_l + u < cnt) {
          // output obase + i + 8 dh: fp16 number (i + 8 dh) of the two runs
          const uint32_t w2 = svw[(i + 8 * dh) >> 1];
          const float sv = __half2float(__ushort_as_half((unsigned short)(i & 1 ? w2 >> 16 : w2 & 0xFFFFu)));
          dst[(size_t)tok_row[u] * p.out + obase + i + 8 * dh] = acc[i][d] * tok_scale[u] * sv;
        }
      }
    item = next_item;
  }
  cp_async_wait<0>();
}

template <int K, int FP8, int HAD>
cudaError_t launch_gemv(const GemvParams& gp, int items_ub, cudaStream_t st) {
  using C = Cfg<K>;
  static int occ = -1, sms = 0;
  auto kfn = gemv_kernel<K, FP8, HAD>;
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
  const int cta_ub = (items_ub + kCW - 1) / kCW;
  if (cta_ub < grid) grid = cta_ub;
  if (grid < 1) grid = 1;
  const cudaError_t err = launch_pdl(kfn, dim3(grid), dim3(kThreads), C::kSmem, st, gp);
  note_launches(1);
  return err;
}

// format v2 (had) rotates in the epilogue: its own instantiations, so the
// format v1 kernels are unchanged by it
template <int HAD>
cudaError_t dispatch_gemv_fmt(int K, int fp8, const GemvParams& gp, int items_ub, cudaStream_t st) {
  if (fp8) {
    if (K == 2) return launch_gemv<2, 1, HAD>(gp, items_ub, st);
    if (K == 3) return launch_gemv<3, 1, HAD>(gp, items_ub, st);
    return launch_gemv<4, 1, HAD>(gp, items_ub, st);
  }
  if (K == 2) return launch_gemv<2, 0, HAD>(gp, items_ub, st);
  if (K == 3) return launch_gemv<3, 0, HAD>(gp, items_ub, st);
  return launch_gemv<4, 0, HAD>(gp, items_ub, st);
}

cudaError_t dispatch_gemv(int K, int fp8, int had, const GemvParams& gp, int items_ub,
                          cudaStream_t st) {
  return had ? dispatch_gemv_fmt<1>(K, fp8, gp, items_ub, st)
             : dispatch_gemv_fmt<0>(K, fp8, gp, items_ub, st);
}

// K splits: the largest power of two (at most 16, keeping >= 8 blocks per
// item, more than any ring is deep) that keeps the expected items at or
// below 4.5 per resident warp (2 CTAs of 8 warps on 152 SMs).  The expected
// token groups are the expected distinct experts of P pairs over E experts,
// E (1 - exp(-P / E)).  Measured on the decode (T 4) and verify (T 32)
// layers: 3-4 items per warp balance the per-item overhead (prologue,
// epilogue, partial rows) against the tail of the dynamic schedule.
int choose_nsplit(size_t P, int E, int items_per_group, int nblk) {
  const double groups = (double)E * (1.0 - exp(-(double)P / (double)E));
  const double cap = 4.5 * 152 * 2 * kCW;
  int ns = 1;
  while (ns < 16 && nblk % (2 * ns) == 0 && nblk / (2 * ns) >= 8 &&
         groups * items_per_group * (2 * ns) <= cap)
    ns *= 2;
  return ns;
}

size_t al(size_t b) { return (b + 255) & ~(size_t)255; }

// Threads of an input pass over n inputs: one per 16-input block, at most
// 256, and at least one full warp (block_max reduces whole warps; blocks
// beyond n/16 idle).  n/16 is a multiple of 8, so every 8-thread rotation
// group is entirely inside or outside the blocks.
int input_pass_threads(int n) {
  const int b = n / 16;
  return b < 32 ? 32 : (b > 256 ? 256 : b);
}

struct GemvLayout {
  size_t xs_gu, xs_gu_inv, gu, xs_d, xs_d_inv, r, counters, entries, total;
  int ns_gu, ns_d;
};

GemvLayout gemv_layout(int T, int top_k, int E, int H, int I) {
  GemvLayout g{};
  const size_t P = (size_t)T * top_k;
  const size_t G = max_groups(T, E, top_k);
  g.ns_gu = choose_nsplit(P, E, 2 * (I / 128), H / 16);
  g.ns_d = choose_nsplit(P, E, H / 128, I / 16);
  size_t o = 0;
  g.xs_gu = o; o += al(G * 2 * (H / 16) * kXsChunk);
  g.xs_gu_inv = o; o += al(P * 2 * 4);
  g.gu = o; o += al((size_t)g.ns_gu * 2 * P * I * 4);
  g.xs_d = o; o += al(G * (I / 16) * kXsChunk);
  g.xs_d_inv = o; o += al(P * 4);
  g.r = o; o += al((size_t)g.ns_d * P * H * 4);
  g.counters = o; o += al(12 * 4);  // 6 item counters, 6 list lengths
  g.entries = o; o += al(3 * G * 3 * 2 * 4);  // lists of (group, projection) for mixed widths
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
  gb->counters = reinterpret_cast<int32_t*>(q + g.counters);
  gb->n_entries = gb->counters + 6;
  gb->entries = reinterpret_cast<int32_t*>(q + g.entries);
  gb->ns_gu = g.ns_gu;
  gb->ns_d = g.ns_d;
}

cudaError_t launch_moe_gemv(const LayerView& L, const void* x, int x_bf16, int T, int top_k,
                            const RouteBuffers& rb, const GemvBuffers& gb, const cudaEvent_t* ev,
                            Shard sh, cudaStream_t st) {
  auto rec = [&](int i) {
    if (ev && ev[i]) record_stage_event(ev[i], st);
  };
  const int P = T * top_k;
  const size_t G = max_groups(T, L.E, top_k);
  cudaError_t err;
  // gather_xs_kernel clears the work counters, except with mixed widths,
  // whose list kernel counts into the same words before it
  if (L.mixed) {
    if ((err = cudaMemsetAsync(gb.counters, 0, 12 * sizeof(int32_t), st)) != cudaSuccess) return err;
    const int threads = (int)(3 * G);
    err = launch_pdl(width_lists_kernel, dim3((unsigned)((threads + 255) / 256)), dim3(256), 0, st,
                     (const int32_t*)(rb.group_off + L.E), (const int32_t*)rb.groups, L.d_kt,
                     (int)(2 * G), (int)G, sh, gb.n_entries, gb.entries);
    note_launches(1);
    if (err != cudaSuccess) return err;
  }
  err = launch_pdl(gather_xs_kernel, dim3(P), dim3(input_pass_threads(L.H)), 0, st, x,
                   x_bf16, L.H, top_k, rb, L.suh[0], L.suh[1], L.had, L.act8, sh, gb.xs_gu,
                   gb.xs_gu_inv, L.mixed ? (int32_t*)nullptr : gb.counters);
  note_launches(1);
  if (err != cudaSuccess) return err;
  rec(2);

  // gate and up share one launch (one per width when the layer mixes widths)
  GemvParams gu{};
  gu.codes[0] = L.codes[0]; gu.codes[1] = L.codes[1];
  gu.stride[0] = L.code_stride[0]; gu.stride[1] = L.code_stride[1];
  gu.in = L.H; gu.out = L.I; gu.nproj = 2; gu.mult = L.mult;
  gu.svh[0] = L.svh[0]; gu.svh[1] = L.svh[1];
  gu.xs = gb.xs_gu; gu.xs_inv = gb.xs_gu_inv;
  // the call's groups: those of experts e0 .. e1 - 1 (groups are in expert order)
  gu.groups = rb.groups; gu.g_begin = rb.group_off + sh.e0; gu.n_groups = rb.group_off + sh.e1;
  gu.seg_pairs = rb.seg_pairs; gu.wts = rb.w; gu.gu_out = gb.gu; gu.n_pos = (size_t)P;
  gu.work = gb.counters; gu.nsplit = gb.ns_gu; gu.proj0 = 0;
  const int ub_gu = (int)(G * 2 * (L.I / 128) * gu.nsplit);
  if (!L.mixed) {
    if ((err = dispatch_gemv(L.K[0], L.fp8, L.had, gu, ub_gu, st)) != cudaSuccess) return err;
  } else {
    // one launch per width over its list (an empty list ends at once)
    gu.off = L.d_off;
    for (int w = 0; w < 3; w++) {
      if (!((L.wmask[0] >> w) & 1)) continue;  // no expert has this width
      GemvParams gw = gu;
      gw.entries = gb.entries + (size_t)w * 2 * G * 2;
      gw.n_entries = gb.n_entries + w;
      gw.work = gb.counters + w;
      if ((err = dispatch_gemv(w + 2, L.fp8, L.had, gw, ub_gu, st)) != cudaSuccess) return err;
    }
  }
  rec(3);

  err = launch_pdl(prep_down_kernel, dim3(P), dim3(input_pass_threads(L.I)), 0, st, gb.gu,
                   gb.ns_gu, (size_t)P, L.I, rb, L.suh[2], L.had, L.act8, sh, gb.xs_d, gb.xs_d_inv);
  note_launches(1);
  if (err != cudaSuccess) return err;
  rec(4);

  GemvParams dn{};
  dn.codes[0] = L.codes[2]; dn.stride[0] = L.code_stride[2];
  dn.in = L.I; dn.out = L.H; dn.nproj = 1; dn.mult = L.mult;
  dn.svh[0] = L.svh[2];
  dn.xs = gb.xs_d; dn.xs_inv = gb.xs_d_inv;
  dn.groups = rb.groups; dn.g_begin = rb.group_off + sh.e0; dn.n_groups = rb.group_off + sh.e1;
  dn.seg_pairs = rb.seg_pairs; dn.wts = rb.w; dn.r_out = gb.r; dn.n_pos = (size_t)P;
  dn.work = gb.counters + 3; dn.nsplit = gb.ns_d; dn.proj0 = 2;
  const int ub_d = (int)(G * (L.H / 128) * dn.nsplit);
  if (!L.mixed) {
    err = dispatch_gemv(L.K[2], L.fp8, L.had, dn, ub_d, st);
  } else {
    dn.off = L.d_off;
    for (int w = 0; w < 3 && err == cudaSuccess; w++) {
      if (!((L.wmask[1] >> w) & 1)) continue;
      GemvParams gw = dn;
      gw.entries = gb.entries + ((size_t)3 * 2 * G + (size_t)w * G) * 2;
      gw.n_entries = gb.n_entries + 3 + w;
      gw.work = gb.counters + 3 + w;
      err = dispatch_gemv(w + 2, L.fp8, L.had, gw, ub_d, st);
    }
  }
  rec(5);
  return err;
}

}  // namespace exl3
