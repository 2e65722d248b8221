// Grouped GEMM path for prefill-sized steps on the 5th-generation tensor
// cores (tcgen05 + TMEM + TMA), with the trellis decoded into shared memory.
//
// Page "GLM-5.3 Flash EXL3 for 2x DGX Sparks", section Cold prefill (E3):
// three GPU-driven launches per MoE layer (gather; gate/up + SwiGLU; down +
// scatter) built from device-side segment tables.  Page "GLM-5.3-Flash ·
// exlr8 (K2/K3/K4)", Widths: with the E4M3 codebook, prefill runs on the
// tensor cores.
//
// One CTA = (token tile of <= 512 positions of one expert, projection,
// 128-output strip).  D[o][n] = sum_i W[i][o] x[n][i] with A = decoded
// weights (M = 128 outputs, MN-major in shared memory) and B = activation rows
// (N = tokens, K-major, loaded by TMA with 128-byte swizzle; each CTA loads
// its own boxes, the neighbouring strips' loads mostly hit L2); fp16 or E4M3
// operands (kind::f16 or kind::f8f6f4), fp32 accumulators in TMEM: two
// 256-column accumulators, so every decoded weight serves up to 512 tokens.
//   warps 0..kDec-1  decode: they take the tile's 16-input blocks
//              round-robin (block j = warp + n kDec), load a block's code row
//              one job ahead into registers (pulled into L2 4 jobs ahead),
//              hash each 32-bit window once, sum the codebook halves into
//              fp16 (E4M3 rule if set), apply suh (fp16 operands, format v1)
//              or keep E4M3 bytes (FP8 operands), and store 16-byte chunks
//              into the swizzled A stage;
//   warp kDec  TMA producer of the B stages, and TMEM allocator;
//   warp kDec+1  one thread issues tcgen05.mma and commits stage releases.
// The epilogue (the decoder warps) reads TMEM: gate/up launch -> svh * acc per
// position, or, fused (format v1, fp16 operands, one width), gate and up of
// the same 64 outputs in one CTA (A rows 0-63 and 64-127) and h = silu(g) u
// written as fp16; down launch -> router weight * svh * acc into the pair's
// own row (no atomics).  Every pipeline wait is bounded; a role whose wait
// gives up stops issuing and unwinds (see pipe_wait).
//
// Format v2 (Hadamard rotation) and FP8 operands: suh cannot be folded into
// the weights (the rotation sits between it and the codes; an E4M3 value
// times suh is no E4M3 value), so the input passes apply it (and rotate each
// 128-input block), gate and up have separate activation rows ([P + pos] for
// up), and the h pass runs after the gate/up launch; the format v2 epilogue
// rotates each 128-output block through shared memory before svh.
#include <cuda.h>

#include "common.cuh"
#include "internal.h"
#include "pipeline.cuh"
#include "umma.cuh"

namespace exl3 {

namespace {

constexpr int kHalfN = 256;           // tokens per TMEM accumulator (MMA N)
constexpr int kBN = 2 * kHalfN;       // tokens per tile
constexpr int kRow = 128;             // bytes of one K step of a K-major operand row
constexpr int kAStages = 5;           // A ring: decoders up to 5 K steps ahead
constexpr int kAStage = 128 * kRow;           // 16 KB: 128 outputs x one K step
constexpr int kBox = 64 * kRow;               // one TMA box: 64 tokens x one K step, 8 KB
constexpr int kBStages = 2;
constexpr int kBStage = kBN * kRow;           // 64 KB
constexpr int kSDec = 16;                     // decoder warps of the small-tile kernel

// Operand element type of the tensor-core kernels: fp16 (kind::f16) or E4M3
// (kind::f8f6f4, the FP8 x FP8 product).  A K step is one 128-byte row of a
// K-major operand either way (64 fp16 or 128 E4M3 inputs), so every stage,
// box and descriptor offset in bytes is the same for both.
template <int OP8>
struct OpT {
  static constexpr int kKS = OP8 ? 128 : 64;           // inputs per K step
  static constexpr int kBlk = 16 * 128 * (OP8 ? 1 : 2);  // one 16-input block of a 128-output tile
  static constexpr int kJobs = kKS / 16;               // 16-input blocks per K step
  static constexpr int kDec = 16;                      // decoder warps (big tiles)
  static constexpr int kThreads = (kDec + 2) * 32;
  static constexpr int kSJobs = 2 * kJobs;             // small tiles: blocks x 2 code strips
  static constexpr int kSPar = kSDec / kSJobs;
};

template <int K>
struct GCfg {
  static constexpr int kCodeChunk = 8 * 32 * K;  // code bytes of one job (8 tiles)
  static constexpr int kOffB = kAStages * kAStage;
  static constexpr int kOffScal = kOffB + kBStages * kBStage;
  static constexpr int kOffBar = kOffScal + kBN * 8;  // per-token scale and pair id
  static constexpr int kNumBars = 2 * kAStages + 2 * kBStages + 1;
  static constexpr int kSmem = kOffBar + kNumBars * 8 + 16 + 1024;  // + alignment slack
};

struct GemmParams {
  const uint16_t* codes[2];
  size_t stride[2];         // uint16 words per expert
  const uint16_t* suh[2];   // [E][in]
  const uint16_t* svh[2];   // [E][out]
  int in, out, nproj;
  uint32_t mult;
  const int32_t* tiles;     // [t][4] {expert, pos0, count, 0}
  const int32_t* n_tiles;
  const float* xinv;        // [pos] scale of the B rows
  float* gu_out;            // gate/up launch: [proj][pos][out]
  size_t n_pos;
  float* r_out;             // down launch: [pair id][out]
  const int32_t* seg_pairs;
  const float* wts;
  int32_t* status;
  long long budget;         // clock budget of every pipeline wait
  int fault_ks;             // test hook: the K step whose operand loads the TMA
                            // thread skips (a wait that nothing completes); -1 = none
  int had;                  // format v2: suh on the activation side, outputs rotated
  int xrow_off;             // activation row (and scale) offset of projection 1
  // mixed widths: this launch's list of (tile, projection) pairs whose width
  // is this instantiation's K, and the experts' code offsets
  const int32_t* entries;   // [n][2], or null: every tile, every projection
  const int32_t* n_entries;
  const unsigned long long* off;  // [E][3] code word offsets, or null: stride * e
  int proj0;                // global index of this launch's projection 0 (0 or 2)
  // SwiGLU in the gate/up epilogue (format v1, fp16 operands, one width):
  // each CTA holds gate and up of the same outputs and writes fp16 h
  int fused;
  uint16_t* h_out;          // [pos][out] fp16 h, times 2^e of its row
  float* hinv;              // [pos] 2^-e (a power of two), written by the chunk-0 CTAs
  const float* hb;          // [E] bound on |h| / |x_t|_1^2 per expert
  const float* l1;          // [T] |x_t|_1
  int top_k;                // pairs per token (position -> token)
};

// Fused SwiGLU: the power-of-two scale 2^e of position pos's h row, from the
// bound hb[e] |x_t|_1^2 on |h| (see side_bound_kernel): the bound times 2^e
// stays below 2^15, so fp16 h never overflows; a power-of-two scale does not
// change the relative rounding of normal fp16 values.
__device__ __forceinline__ float h_row_scale(const GemmParams& p, int e, int pos) {
  const float l = p.l1[p.seg_pairs[pos] / p.top_k];
  const float bound = p.hb[e] * l * l;
  int eh = 0;
  if (!isfinite(bound)) eh = -100;
  else if (bound > 0.0f) eh = 14 - ilogbf(bound);
  eh = eh < -100 ? -100 : (eh > 100 ? 100 : eh);
  return ldexpf(1.0f, eh);
}

// (tile, projection) of the CTA's work unit u (its index over strips): from
// the width's list in mixed mode, else u = tile * nproj + projection.  False
// past the end of the work.
__device__ __forceinline__ bool tile_of(const GemmParams& p, int u, int* tile, int* pj) {
  if (p.entries) {
    if (u >= p.n_entries[0]) return false;
    *tile = p.entries[2 * u];
    *pj = p.entries[2 * u + 1];
    return true;
  }
  *pj = u % p.nproj;
  *tile = u / p.nproj;
  return *tile < p.n_tiles[0];
}

// First code word of projection pj of expert e.
__device__ __forceinline__ const uint16_t* gemm_expert_codes(const GemmParams& p, int e, int pj) {
  return (pj ? p.codes[1] : p.codes[0]) +
         (p.off ? (size_t)p.off[(size_t)e * 3 + p.proj0 + pj]
                : (pj ? p.stride[1] : p.stride[0]) * (size_t)e);
}

__device__ __forceinline__ float warp_max(float v) {
  for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
  return v;
}

// 8 activations (fp16 or bf16 bits) as floats.
__device__ __forceinline__ void act8(const uint4& r, int bf16, float (&f)[8]) {
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

__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
  const __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Pipeline wait of one CTA role.  A false return means: stop issuing work
// and unwind.  It happens when this wait ran out of budget, when any CTA of
// the grid recorded a timeout (status bit 4), or when another role of this
// CTA already gave up (abort flag in shared memory); in every case bit 4 of
// the status word is set by the time any role sees the false return.
__device__ __forceinline__ bool pipe_wait(uint64_t* bar, uint32_t parity, const GemmParams& p,
                                          volatile uint32_t* abort_flag) {
  if (*abort_flag) return false;
  if (mbar_wait_or_abort(bar, parity, p.status, p.budget)) return true;
  *abort_flag = 1;
  return false;
}

// Epilogue entry of the decoder warps (threads 0 .. nthreads - 1): wait for
// the accumulator, then take one CTA-wide decision whether to read TMEM and
// store (thread 0 decides between two named barriers), so that warps which
// exchange data through named barriers in the epilogue all take the same
// branch.  False once any role of the grid gave up.
constexpr int kEpiBar = 15;  // named barrier id (the epilogues use 1 .. 8)
__device__ __forceinline__ bool epilogue_live(uint64_t* acc_full, const GemmParams& p,
                                              volatile uint32_t* abort_flag,
                                              volatile uint32_t* live_slot, int nthreads) {
  pipe_wait(acc_full, 0, p, abort_flag);
  named_bar_sync(kEpiBar, nthreads);
  if (threadIdx.x == 0)
    *live_slot = !*abort_flag && !(*reinterpret_cast<volatile int32_t*>(p.status) & 4);
  named_bar_sync(kEpiBar, nthreads);
  return *live_slot != 0;
}

// Format v2 epilogue of the M = outputs kernel: the 4 warps of a column group
// hold the 128 outputs of a strip (TMEM lanes, thread = output) for the same
// 16 token columns.  They stage them in shared memory ([output][17] floats,
// conflict free both ways), then each warp takes 4 of the columns with lane l
// holding outputs l + 32 j, rotates (j in registers, l by shuffles), scales
// and stores 128 contiguous outputs of the token's row.
__device__ __forceinline__ void rotate_store_cols(float* xbuf, const float (&a0)[16], int q4,
                                                  int lane, int bar_id, int c0, int cnt,
                                                  const float (&sv)[4], const float* s_scale,
                                                  const int32_t* s_pid, const GemmParams& p,
                                                  int pj, int pos0, int o0) {
#pragma unroll
  for (int i = 0; i < 16; i++) xbuf[(32 * q4 + lane) * 17 + i] = a0[i];
  named_bar_sync(bar_id, 128);
#pragma unroll
  for (int tt = 0; tt < 4; tt++) {
    const int cl = 4 * q4 + tt, n = c0 + cl;
    float v[4];
#pragma unroll
    for (int j = 0; j < 4; j++) v[j] = xbuf[(lane + 32 * j) * 17 + cl];
    wht_regs(v);
#pragma unroll
    for (int m = 1; m < 32; m <<= 1)
#pragma unroll
      for (int j = 0; j < 4; j++) v[j] = wht_lane(v[j], m, 0xffffffffu);
    if (n < cnt) {
      const float sc = s_scale[n];
      float* dst = p.gu_out ? p.gu_out + ((size_t)pj * p.n_pos + pos0 + n) * p.out
                            : p.r_out + (size_t)s_pid[n] * p.out;
#pragma unroll
      for (int j = 0; j < 4; j++) dst[o0 + lane + 32 * j] = v[j] * sc * sv[j];
    }
  }
  named_bar_sync(bar_id, 128);  // the buffer is refilled by the next chunk
}

// {a, b} halves of lane weights u = 16 pp .. 16 pp + 15.  For K = 2 and 4 each
// 32-bit window is hashed once (a sliding window of 16 + 16/K products whose
// tail is carried to the next pp); see lane_halves for the correction.
template <int K, int PP>
__device__ __forceinline__ void halves16(const LaneWords<K>& lw, uint32_t mult, uint32_t neg16,
                                         const McgConsts& mc,
                                         uint32_t (&xp)[16 + (K == 3 ? 0 : 16 / K)],
                                         uint32_t (&m)[16]) {
  if constexpr (K == 3) {
#pragma unroll
    for (int t = 0; t < 16; t++) m[t] = mcg_halves(lane_state<K>(lw, 16 * PP + t), mult, mc);
  } else {
    constexpr int step = 16 / K;
    if constexpr (PP == 0) {
#pragma unroll
      for (int t = 0; t < step; t++) xp[t] = lane_window32<K>(lw, t * K) * mult;
    } else {
#pragma unroll
      for (int t = 0; t < step; t++) xp[t] = xp[16 + t];
    }
#pragma unroll
    for (int t = step; t < 16 + step; t++) xp[t] = lane_window32<K>(lw, (16 * PP + t) * K) * mult;
#pragma unroll
    for (int t = 0; t < 16; t++) m[t] = mcg_maskxor(xp[t + step] * neg16 + xp[t], mc);
  }
}

// Tile (of the 8 in a code row) that lane decodes, quad lane c = lane & 3 of
// it.  Tiles g and g ^ 2 share a quarter warp (lanes 8q .. 8q + 7), so the 8
// lanes of every 16-byte store phase of decode_store land in 8 different
// 16-byte bank groups of the swizzled stage (with g = lane >> 2 the pairs g,
// g ^ 1 collide two ways).
__device__ __forceinline__ int dec_tile(int lane) {
  const int l4 = lane >> 2;
  return (l4 & 4) | ((l4 & 1) << 1) | ((l4 >> 1) & 1);
}

// Decode this lane's 64 weights of one tile and store them into the MN-major
// A stage: lane (g, c) holds outputs 16g..16g+15 (rows of the strip) for
// inputs c, c+4, c+8, c+12 of the block.  off[4hf + 2jh + jl] is the lane's
// byte offset of the 16-byte chunk (input c + 4jh + 8hf, rows 8jl..8jl+7).
template <int K, int FP8>
__device__ __forceinline__ void decode_store(const LaneWords<K>& lw, uint32_t mult, uint32_t neg16,
                                             uint8_t* a_blk, const int (&off)[8],
                                             const uint32_t (&s2)[4]) {
  const McgConsts mc = mcg_consts();
  uint32_t v[8][4];
  uint32_t xp[16 + (K == 3 ? 0 : 16 / K)];
  uint32_t m[16];
#define EXL3_PP(PP)                                                            \
  halves16<K, PP>(lw, mult, neg16, mc, xp, m);                                 \
  _Pragma("unroll") for (int idx = 0; idx < 8; idx++) {                        \
    const int t0 = idx; /* t = 8 rr + 4 hf + 2 jh + jl, rr = 0 */              \
    uint32_t v2 = sum_halves2(m[t0], m[t0 + 8]);                               \
    if (FP8) v2 = e4m3_round2(v2);                                             \
    __half2 hh = __hmul2(*reinterpret_cast<const __half2*>(&v2),               \
                         *reinterpret_cast<const __half2*>(&s2[idx >> 1]));    \
    v[idx][PP] = *reinterpret_cast<uint32_t*>(&hh);                            \
  }
  EXL3_PP(0)
  EXL3_PP(1)
  EXL3_PP(2)
  EXL3_PP(3)
#undef EXL3_PP
#pragma unroll
  for (int idx = 0; idx < 8; idx++)
    *reinterpret_cast<uint4*>(a_blk + off[idx]) = make_uint4(v[idx][0], v[idx][1], v[idx][2], v[idx][3]);
}

// sum_halves2 as two scalar half adds whose operands are the halves of one
// register (selected by the add itself, no permutes) and one pack: the same
// IEEE fp16 round-to-nearest sums with 0.42 fewer ALU-pipe instructions per
// weight in this inner loop (measured; moved to the FMA pipe) but a few more
// live registers.  The E4M3-byte decoders use it; the fp16-operand ones keep
// the permute form (at the small-tile kernel's 96-register cap this form
// spills and measured slower).
__device__ __forceinline__ uint32_t sum_halves2_sel(uint32_t m0, uint32_t m1) {
  const __half2 h0 = *reinterpret_cast<const __half2*>(&m0);
  const __half2 h1 = *reinterpret_cast<const __half2*>(&m1);
  const __half2 r = __halves2half2(__hadd(__low2half(h0), __high2half(h0)),
                                   __hadd(__low2half(h1), __high2half(h1)));
  return *reinterpret_cast<const uint32_t*>(&r);
}

// FP8 operand variant: the lane's 64 weights as E4M3 bytes (the codebook
// value under the E4M3 rule; suh is on the activation side), in four 16-byte
// chunks of the 1-byte MN-major stage, one per input column c + 4jh + 8hf,
// each holding the lane's 16 output rows in order.  off[2hf + jh] is the
// chunk's swizzled byte offset.
template <int K>
__device__ __forceinline__ void decode_store8(const LaneWords<K>& lw, uint32_t mult,
                                              uint32_t neg16, uint8_t* a_blk,
                                              const int (&off)[4]) {
  const McgConsts mc = mcg_consts();
  uint32_t f[8][4];  // [4hf + 2jh + jl][PP]: E4M3 bytes of rows 2PP + 8jl, 2PP + 1 + 8jl
  uint32_t xp[16 + (K == 3 ? 0 : 16 / K)];
  uint32_t m[16];
#define EXL3_PP8(PP)                                                           \
  halves16<K, PP>(lw, mult, neg16, mc, xp, m);                                 \
  _Pragma("unroll") for (int idx = 0; idx < 8; idx++)                         \
      f[idx][PP] = e4m3_bytes2(sum_halves2_sel(m[idx], m[idx + 8]));
  EXL3_PP8(0)
  EXL3_PP8(1)
  EXL3_PP8(2)
  EXL3_PP8(3)
#undef EXL3_PP8
#pragma unroll
  for (int c4 = 0; c4 < 4; c4++) {
    const int i0 = 2 * c4, i1 = 2 * c4 + 1;  // row groups jl = 0 (rows 0..7), 1 (rows 8..15)
    *reinterpret_cast<uint4*>(a_blk + off[c4]) =
        make_uint4(__byte_perm(f[i0][0], f[i0][1], 0x5410), __byte_perm(f[i0][2], f[i0][3], 0x5410),
                   __byte_perm(f[i1][0], f[i1][1], 0x5410), __byte_perm(f[i1][2], f[i1][3], 0x5410));
  }
}

// Lane-to-tile map of the FP8 decoders: each quarter warp holds tiles g and
// g ^ 4, whose 16-byte chunks (chunk index g ^ row) fall in 8 different
// 16-byte bank groups of the 1-byte stage.
__device__ __forceinline__ int dec_tile8(int lane) {
  return ((lane >> 3) & 3) | (((lane >> 2) & 1) << 2);
}

template <int K, int FP8, int OP8>
__global__ void __launch_bounds__(OpT<OP8>::kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmap_b, GemmParams p) {
  using C = GCfg<K>;
  using T = OpT<OP8>;
  constexpr int kDec = T::kDec, kJobs = T::kJobs, kKS = T::kKS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~(uintptr_t)1023);
  // fused gate/up: 64 outputs of each projection per CTA (A rows 0-63 gate,
  // 64-127 up, against the same activation rows)
  const int strips = p.out / (p.fused ? 64 : 128);
  const int s = blockIdx.x % strips;
  pdl_wait();
  int tile, pj;
  if (!tile_of(p, blockIdx.x / strips, &tile, &pj)) return;
  const int e = p.tiles[4 * tile], pos0 = p.tiles[4 * tile + 1], cnt = p.tiles[4 * tile + 2];
  const int n0 = cnt < kHalfN ? ((cnt + 15) / 16) * 16 : kHalfN;
  const int n1 = cnt > kHalfN ? ((cnt - kHalfN + 15) / 16) * 16 : 0;
  const int nbox = (n0 + n1 + 63) / 64;
  constexpr int nbst = kBStages, nast = kAStages;
  const int bstage = kBStage;
  uint8_t* const b_ring = smem + C::kOffB;
  const int nks = p.in / kKS;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* a_full = bars;
  uint64_t* a_empty = a_full + kAStages;
  uint64_t* b_full = a_empty + kAStages;
  uint64_t* b_empty = b_full + kBStages;
  uint64_t* acc_full = b_empty + kBStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 1);
  volatile uint32_t* abort_flag = tmem_slot + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < nast; i++) {
      mbar_init(&a_full[i], kJobs);
      mbar_init(&a_empty[i], 1);
    }
    for (int i = 0; i < nbst; i++) {
      mbar_init(&b_full[i], 1);
      mbar_init(&b_empty[i], 1);
    }
    mbar_init(acc_full, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kDec) tmem_alloc(tmem_slot, 2 * kHalfN);
  // per-token epilogue scalars: scale = 1/row-scale (* router weight), pair id
  float* s_scale = reinterpret_cast<float*>(smem + C::kOffScal);
  int32_t* s_pid = reinterpret_cast<int32_t*>(s_scale + kBN);
  // activation rows (and their scales) of this projection start at xrow0
  const int xrow0 = pj * p.xrow_off + pos0;
  for (int n = threadIdx.x; n < cnt; n += blockDim.x) {
    const int pos = pos0 + n;
    float sc = p.xinv[xrow0 + n];
    int pid = 0;
    if (p.r_out) {  // down launch: the pair's row and router weight
      pid = p.seg_pairs[pos];
      sc *= p.wts[pid];
    } else if (p.fused) {  // fused gate/up: the scale of h's row, 2^e
      const float hs = h_row_scale(p, e, pos);
      if (s == 0) p.hinv[pos] = 1.0f / hs;  // for the down launch
      pid = __float_as_int(hs);
    }
    s_scale[n] = sc;
    s_pid[n] = pid;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kDec) {
    // ---------------------------------------------------------------- TMA
    // The strips of a tile are neighbouring CTAs, so the activation boxes one
    // CTA loads are mostly L2 hits for the others.  (single-thread loops:
    // stage index and phase advance incrementally and the descriptors are
    // precomputed, so nothing on this critical path divides)
    if (lane == 0) {
      int sb = 0, issued = 0;
      uint32_t pb = 0;
      for (int ks = 0; ks < nks; ks++) {
        if (!pipe_wait(&b_empty[sb], pb ^ 1, p, abort_flag)) break;
        if (ks != p.fault_ks) {
          mbar_arrive_expect_tx(&b_full[sb], nbox * kBox);
          uint8_t* dst = b_ring + sb * bstage;
          for (int j = 0; j < nbox; j++)
            tma_load_2d(dst + j * kBox, &tmap_b, ks * kKS, xrow0 + 64 * j, &b_full[sb]);
        }
        issued = ks + 1;
        if (++sb == nbst) {
          sb = 0;
          pb ^= 1;
        }
      }
      // before the CTA may exit, every box this thread requested has landed:
      // loads can be outstanding only in the last nbst stages issued (a stage
      // is refilled only after the MMA consumed it)
      for (int ks = issued - nbst < 0 ? 0 : issued - nbst; ks < issued; ks++)
        if (ks != p.fault_ks) mbar_drain(&b_full[ks % nbst], (ks / nbst) & 1, p.budget);
    }
  } else if (warp == kDec + 1) {
    // ---------------------------------------------------------------- MMA
    if (lane == 0) {
      const uint32_t id0 = umma_idesc_f16(128, n0, 1, 0);
      const uint32_t id1 = umma_idesc_f16(128, n1 > 0 ? n1 : 16, 1, 0);
      // descriptor address fields are byte addresses >> 4 (no carry below
      // 256 KB), so stage and K-slice offsets are plain additions
      // A (decoded weights, MN-major): fp16 rows hold 64 outputs (two atoms
      // 1024 B apart, 8-input groups 2048 B apart); E4M3 rows hold all 128
      // (one atom, 8-input groups 1024 B apart)
      const uint64_t a_desc0 = umma_desc(smem_u32(smem), 1024, OP8 ? 1024 : 2048);
      const uint64_t b_desc0 = umma_desc(smem_u32(b_ring), 16, 1024);
      int sa = 0, sb = 0;
      uint32_t pa = 0, pb = 0;
      for (int ks = 0; ks < nks; ks++) {
        if (!pipe_wait(&a_full[sa], pa, p, abort_flag) || !pipe_wait(&b_full[sb], pb, p, abort_flag))
          break;
        tc_fence_after();
        const uint64_t ad = a_desc0 + (uint64_t)(sa * (kAStage >> 4));
        const uint64_t bd = b_desc0 + (uint64_t)(sb * (bstage >> 4));
#pragma unroll
        for (int kk = 0; kk < 4; kk++) {  // K slices of 32 bytes
          const uint32_t acc = (ks > 0 || kk > 0) ? 1u : 0u;
          if (OP8) {
            umma_e4m3(tmem, ad + kk * (4096 >> 4), bd + kk * (32 >> 4), id0, acc);
            if (n1 > 0)
              umma_e4m3(tmem + kHalfN, ad + kk * (4096 >> 4),
                        bd + ((kHalfN * 128) >> 4) + kk * (32 >> 4), id1, acc);
          } else {
            umma_f16(tmem, ad + kk * (4096 >> 4), bd + kk * (32 >> 4), id0, acc);
            if (n1 > 0)
              umma_f16(tmem + kHalfN, ad + kk * (4096 >> 4),
                       bd + ((kHalfN * 128) >> 4) + kk * (32 >> 4), id1, acc);
          }
        }
        umma_commit(&a_empty[sa]);
        umma_commit(&b_empty[sb]);
        if (++sa == nast) {
          sa = 0;
          pa ^= 1;
        }
        if (++sb == nbst) {
          sb = 0;
          pb ^= 1;
        }
      }
      // always committed, after an abort too: it completes once every MMA
      // issued above is done, which TMEM deallocation waits for
      umma_commit(acc_full);
    }
  } else {
    // ---------------------------------------------------------------- decode
    // jobs are the tile's 16-input blocks j = 0 .. nks * kJobs - 1 (K step
    // j / kJobs, block j % kJobs of it); warp w takes j = w, w + kDec, ...
    const int g = OP8 ? dec_tile8(lane) : dec_tile(lane), c = lane & 3;
    const size_t row_bytes = (size_t)(p.out / 16) * 32 * K;
    // this lane's tile: tile g of the strip, or (fused) tile g & 3 of the
    // 64-output chunk of gate (g < 4) or up (g >= 4)
    const int pg = p.fused ? g >> 2 : pj;
    const int tcol = p.fused ? 4 * s + (g & 3) : 8 * s + g;
    const uint8_t* lbase = reinterpret_cast<const uint8_t*>(gemm_expert_codes(p, e, pg)) +
                           ((size_t)tcol * 4 + c) * 8 * K;
    // the 16-input block rows this warp pulls into L2: one strip, or (fused)
    // the gate half (lanes 0-15) and the up half (lanes 16-31)
    const int lpf = p.fused ? lane & 15 : lane;
    const uint8_t* pbase =
        reinterpret_cast<const uint8_t*>(gemm_expert_codes(p, e, p.fused ? lane >> 4 : pj)) +
        (size_t)(p.fused ? 4 * s : 8 * s) * 32 * K + lpf * 128;
    const int pf_bytes = (p.fused ? 4 : 8) * 32 * K;
    const int n_jobs = nks * kJobs;
    const int n_my = warp < n_jobs ? (n_jobs - warp + kDec - 1) / kDec : 0;
    // lane-constant swizzled offsets of this lane's output chunks in a block:
    // fp16, 8 chunks of 8 outputs (input c + 4jh + 8hf, rows 8jl..8jl+7);
    // E4M3, 4 chunks of 16 outputs (input c + 4jh + 8hf)
    int off[8], off8[4];
#pragma unroll
    for (int idx = 0; idx < 8; idx++) {
      const int hf = idx >> 2, jh = (idx >> 1) & 1, jl = idx & 1;
      const int kr = c + 4 * jh;  // input row inside its 8-row K group
      off[idx] = (g >> 2) * 1024 + hf * 2048 + kr * 128 + (((2 * (g & 3) + jl) ^ kr) << 4);
    }
#pragma unroll
    for (int c4 = 0; c4 < 4; c4++) {
      const int hf = c4 >> 1, kr = c + 4 * (c4 & 1);
      off8[c4] = hf * 1024 + kr * 128 + ((g ^ kr) << 4);
    }
    const uint32_t neg16 = opaque_u32(0xFFFF0000u);
    // this lane's 8K code bytes of job n (code lane `lane` of the 8-tile
    // chunk); the code row of block j of the tile is row j of the expert
    auto lane_codes = [&](int n) {
      const int j = warp + n * kDec;
      return reinterpret_cast<const uint16_t*>(lbase + (size_t)j * row_bytes);
    };
    // code rows are pulled into L2 kL2Ahead jobs ahead, so the register
    // prefetch one job ahead hits L2 (a measured sweep: 4 jobs beat 2, 8
    // and 16)
    constexpr int kL2Ahead = 4;
    auto prefetch_l2 = [&](int n) {
      if (n < n_my && lpf * 128 < pf_bytes) {
        const uint8_t* a = pbase + (size_t)(warp + n * kDec) * row_bytes;
        asm volatile("prefetch.global.L2 [%0];" ::"l"(a));
      }
    };
    for (int n = 0; n < kL2Ahead; n++) prefetch_l2(n);
    const uint16_t* suh_e = (pg ? p.suh[1] : p.suh[0]) + (size_t)e * p.in + c;
    // suh of this lane's 4 inputs of a block (inputs 16 j + c + 4 jh + 8 hf),
    // loaded one job ahead
    uint32_t s2n[4];
    auto load_suh = [&](int n) {
      const int j = warp + n * kDec;
#pragma unroll
      for (int q = 0; q < 4; q++)  // format v2, FP8 operands: suh is on the activation side
        s2n[q] = p.had || OP8 ? 0x3C00u : __ldg(suh_e + 16 * j + 4 * (q & 1) + 8 * (q >> 1));
    };
    LaneWords<K> nxt;
    if (n_my > 0) {
      load_suh(0);
      load_lane_words<K>(nxt, lane_codes(0));
    }
    for (int n = 0; n < n_my; n++) {
      const int j = warp + n * kDec, ks = j / kJobs, blk = j % kJobs;
      const int sa = ks % nast;                      // the K step's A stage
      const uint32_t pa = (uint32_t)(ks / nast) & 1u;  // and its fill count's parity
      LaneWords<K> lw = nxt;
      if (n + 1 < n_my) load_lane_words<K>(nxt, lane_codes(n + 1));
      prefetch_l2(n + kL2Ahead);
      uint32_t s2[4];
#pragma unroll
      for (int q = 0; q < 4; q++) s2[q] = s2n[q] | (s2n[q] << 16);
      if (n + 1 < n_my) load_suh(n + 1);
      fetch_neighbour<K>(lw);
      if (!__all_sync(0xffffffffu, pipe_wait(&a_empty[sa], pa ^ 1, p, abort_flag))) break;
      if (OP8)
        decode_store8<K>(lw, p.mult, neg16, smem + sa * kAStage + blk * T::kBlk, off8);
      else
        decode_store<K, FP8>(lw, p.mult, neg16, smem + sa * kAStage + blk * T::kBlk, off, s2);
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&a_full[sa]);
    }

    // ------------------------------------------------------------- epilogue
    // (skipped, stores and all, once any role of the grid gave up)
    const bool live = epilogue_live(acc_full, p, abort_flag, abort_flag + 1, kDec * 32);
    tc_fence_after();
    // warp w reads TMEM lanes 32 (w % 4) .. + 31 (its access quarter) and
    // every (kDec/4)-th chunk of 16 token columns (column n = token n: the
    // second accumulator starts at column kHalfN)
    const int q4 = warp & 3, cgrp = warp >> 2;
    const int o = 128 * s + 32 * q4 + lane;
    const uint32_t trow = tmem + ((uint32_t)(32 * q4) << 16);
    const uint16_t* svh_e = (pj ? p.svh[1] : p.svh[0]) + (size_t)e * p.out;
    if (live && p.fused) {
      // SwiGLU: TMEM lanes 0-63 hold gate outputs 0-63 of the 64-output
      // chunk, lanes 64-127 the up outputs of the same channels.  Per 16
      // token columns the 4 warps of a column group stage their scaled
      // values in shared memory (the A ring is idle; [row][17] floats,
      // conflict free both ways); then each warp takes 4 of the columns, lane
      // l forms h = silu(g) u for channels l and l + 32, scales it by the
      // row's 2^e and the warp stores 64 consecutive fp16 outputs per token.
      float* xbuf = reinterpret_cast<float*>(smem) + cgrp * (128 * 17);
      const int row = 32 * q4 + lane;  // TMEM lane = A row
      const float svf = __half2float(__ushort_as_half(
          p.svh[q4 >> 1][(size_t)e * p.out + 64 * s + (row & 63)]));
      for (int c0 = 16 * cgrp; c0 < cnt; c0 += 16 * (kDec / 4)) {
        float a0[16];
        tmem_ld16(trow + c0, a0);
        tmem_ld_wait(a0);
#pragma unroll
        for (int i = 0; i < 16; i++) xbuf[row * 17 + i] = a0[i] * svf;
        named_bar_sync(1 + cgrp, 128);
#pragma unroll
        for (int tt = 0; tt < 4; tt++) {
          const int cl = 4 * q4 + tt, n = c0 + cl;
          if (n < cnt) {
            const float sc = s_scale[n], hsc = __int_as_float(s_pid[n]);
            uint16_t* dst = p.h_out + (size_t)(pos0 + n) * p.out + 64 * s;
#pragma unroll
            for (int hh = 0; hh < 2; hh++) {
              const int ch = lane + 32 * hh;
              const float gv = xbuf[ch * 17 + cl] * sc, uv = xbuf[(64 + ch) * 17 + cl] * sc;
              dst[ch] = __half_as_ushort(__float2half_rn(silu_f(gv) * uv * hsc));
            }
          }
        }
        named_bar_sync(1 + cgrp, 128);  // the buffer is refilled by the next chunk
      }
    }
    if (live && p.had) {
      // the A ring is idle once the accumulator is complete
      float* xbuf = reinterpret_cast<float*>(smem) + cgrp * (128 * 17);
      float svr[4];
#pragma unroll
      for (int j = 0; j < 4; j++)
        svr[j] = __half2float(__ushort_as_half(svh_e[128 * s + lane + 32 * j]));
      for (int c0 = 16 * cgrp; c0 < cnt; c0 += 16 * (kDec / 4)) {
        float a0[16];
        tmem_ld16(trow + c0, a0);
        tmem_ld_wait(a0);
        rotate_store_cols(xbuf, a0, q4, lane, 1 + cgrp, c0, cnt, svr, s_scale, s_pid, p, pj, pos0,
                          128 * s);
      }
    }
    const float sv = __half2float(__ushort_as_half(svh_e[o]));
    for (int c0 = p.had || p.fused || !live ? cnt : 16 * cgrp; c0 < cnt; c0 += 16 * (kDec / 4)) {
      float a0[16];
      tmem_ld16(trow + c0, a0);
      tmem_ld_wait(a0);
#pragma unroll
      for (int i = 0; i < 16; i++) {
        const int n = c0 + i;
        if (n < cnt) {
          const float v = a0[i] * s_scale[n] * sv;
          if (!p.r_out)
            p.gu_out[((size_t)pj * p.n_pos + pos0 + n) * p.out + o] = v;
          else
            p.r_out[(size_t)s_pid[n] * p.out + o] = v;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kDec) {
    // every MMA issued has completed (immediate unless a role gave up early)
    mbar_drain(acc_full, 0, p.budget);
    tc_fence_after();
    tmem_dealloc(tmem, 2 * kHalfN);
  }
}

// ---------------------------------------------------------------------------
// Small-tile variant (tiles of <= 128 tokens).  The tensor core's cost per
// instruction is nearly flat up to N = 128, so for a tile this small the
// operands are swapped: D[token][output] = sum_i x[token][i] W[i][output] with
// A = the activation rows (M = 64 or 128 tokens, K-major, TMA) and B = the
// decoded weights (N = 256 outputs, MN-major): one instruction covers 2x (M 64)
// or 4x (M 128) the weights of the M = 128 / N = 64 form.  One CTA = (tile,
// projection, 256 outputs = two code strips); 16 decoder warps (two K steps
// in flight), one TMA warp, one MMA warp.  The accumulator holds, per TMEM
// lane quarter q, tokens 16q + i (M 64, lanes 32q + i, i < 16) or 32q + i
// (M 128); column = output.
constexpr int kSN = 256;                       // outputs per CTA (MMA N)
constexpr int kSM = 128;                       // tokens at most (MMA M 64 or 128)
constexpr int kSThreads = (kSDec + 2) * 32;    // kSDec decoder warps, TMA, MMA
constexpr int kSWStages = 5;                   // decoded-weight stages
constexpr int kSWStage = kSN * kRow;           // 32 KB
constexpr int kSXStages = 4;                   // activation stages
constexpr int kSXStage = kSM * kRow;           // 16 KB (M 64 uses the first half)

struct SCfg {
  static constexpr int kOffX = kSWStages * kSWStage;
  static constexpr int kOffScal = kOffX + kSXStages * kSXStage;
  static constexpr int kOffBar = kOffScal + kSM * 8;
  static constexpr int kNumBars = 2 * kSWStages + 2 * kSXStages + 1;
  static constexpr int kSmem = kOffBar + kNumBars * 8 + 16 + 1024;
};
static_assert(SCfg::kSmem <= 227 * 1024, "small-tile kernel shared memory");

template <int K, int FP8, int OP8>
__global__ void __launch_bounds__(kSThreads, 1)
    gemm64_kernel(const __grid_constant__ CUtensorMap tmap_x, GemmParams p) {
  using T = OpT<OP8>;
  constexpr int kSJobs = T::kSJobs, kSPar = T::kSPar, kKS = T::kKS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~(uintptr_t)1023);
  // fused gate/up: 128 outputs of each projection per CTA (B columns 0-127
  // gate, 128-255 up)
  const int chunks = p.out / (p.fused ? kSN / 2 : kSN);
  const int s = blockIdx.x % chunks;
  pdl_wait();
  int tile, pj;
  if (!tile_of(p, blockIdx.x / chunks, &tile, &pj)) return;
  const int e = p.tiles[4 * tile], pos0 = p.tiles[4 * tile + 1], cnt = p.tiles[4 * tile + 2];
  const int nks = p.in / kKS;
  const int tm = cnt <= 64 ? 64 : 128;  // MMA M
  const int nxbox = tm / 64;            // 64-token boxes per activation stage

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SCfg::kOffBar);
  uint64_t* w_full = bars;
  uint64_t* w_empty = w_full + kSWStages;
  uint64_t* x_full = w_empty + kSWStages;
  uint64_t* x_empty = x_full + kSXStages;
  uint64_t* acc_full = x_empty + kSXStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 1);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  uint8_t* const x_ring = smem + SCfg::kOffX;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kSWStages; i++) {
      mbar_init(&w_full[i], kSJobs);
      mbar_init(&w_empty[i], 1);
    }
    for (int i = 0; i < kSXStages; i++) {
      mbar_init(&x_full[i], 1);
      mbar_init(&x_empty[i], 1);
    }
    mbar_init(acc_full, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kSDec) tmem_alloc(tmem_slot, kSN);
  float* s_scale = reinterpret_cast<float*>(smem + SCfg::kOffScal);
  int32_t* s_pid = reinterpret_cast<int32_t*>(s_scale + kSM);
  // activation rows (and their scales) of this projection start at xrow0
  const int xrow0 = pj * p.xrow_off + pos0;
  for (int n = threadIdx.x; n < cnt; n += blockDim.x) {
    const int pos = pos0 + n;
    float sc = p.xinv[xrow0 + n];
    int pid = 0;
    if (p.r_out) {  // down launch: the pair's row and router weight
      pid = p.seg_pairs[pos];
      sc *= p.wts[pid];
    } else if (p.fused) {  // fused gate/up: the scale of h's row, 2^e
      const float hs = h_row_scale(p, e, pos);
      if (s == 0) p.hinv[pos] = 1.0f / hs;  // for the down launch
      pid = __float_as_int(hs);
    }
    s_scale[n] = sc;
    s_pid[n] = pid;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kSDec) {
    // ---------------------------------------------------------------- TMA
    // one or two 64-token boxes per K step (the output chunks of a tile are
    // neighbouring CTAs, so most of these loads hit L2)
    if (lane == 0) {
      int sx = 0, issued = 0;
      uint32_t px = 0;
      for (int ks = 0; ks < nks; ks++) {
        if (!pipe_wait(&x_empty[sx], px ^ 1, p, abort_flag)) break;
        if (ks != p.fault_ks) {
          mbar_arrive_expect_tx(&x_full[sx], nxbox * kBox);
          for (int j = 0; j < nxbox; j++)
            tma_load_2d(x_ring + sx * kSXStage + j * kBox, &tmap_x, ks * kKS, xrow0 + 64 * j,
                        &x_full[sx]);
        }
        issued = ks + 1;
        if (++sx == kSXStages) {
          sx = 0;
          px ^= 1;
        }
      }
      // drain: loads can be outstanding only in the last kSXStages issued
      for (int ks = issued - kSXStages < 0 ? 0 : issued - kSXStages; ks < issued; ks++)
        if (ks != p.fault_ks)
          mbar_drain(&x_full[ks % kSXStages], (ks / kSXStages) & 1, p.budget);
    }
  } else if (warp == kSDec + 1) {
    // ---------------------------------------------------------------- MMA
    if (lane == 0) {
      // A: activations K-major (8-row atoms 1024 B apart, K slice +32 B);
      // B: decoded weights MN-major (64-output atoms 1024 B apart, 8-input
      // groups 4096 B apart, K slice of 16 = +8192 B)
      const uint32_t idesc = umma_idesc_f16(tm, kSN, 0, 1);
      const uint64_t x_desc0 = umma_desc(smem_u32(x_ring), 16, 1024);
      // E4M3 rows hold 128 outputs: two atoms, 8-input groups 2048 B apart
      const uint64_t w_desc0 = umma_desc(smem_u32(smem), 1024, OP8 ? 2048 : 4096);
      int sw = 0, sx = 0;
      uint32_t pw = 0, px = 0;
      for (int ks = 0; ks < nks; ks++) {
        if (!pipe_wait(&w_full[sw], pw, p, abort_flag) || !pipe_wait(&x_full[sx], px, p, abort_flag))
          break;
        tc_fence_after();
        const uint64_t xd = x_desc0 + (uint64_t)(sx * (kSXStage >> 4));
        const uint64_t wd = w_desc0 + (uint64_t)(sw * (kSWStage >> 4));
#pragma unroll
        for (int kk = 0; kk < 4; kk++) {  // K slices of 32 bytes
          if (OP8)
            umma_e4m3(tmem, xd + kk * (32 >> 4), wd + kk * (8192 >> 4), idesc,
                      (ks > 0 || kk > 0) ? 1u : 0u);
          else
            umma_f16(tmem, xd + kk * (32 >> 4), wd + kk * (8192 >> 4), idesc,
                     (ks > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(&w_empty[sw]);
        umma_commit(&x_empty[sx]);
        if (++sw == kSWStages) {
          sw = 0;
          pw ^= 1;
        }
        if (++sx == kSXStages) {
          sx = 0;
          px ^= 1;
        }
      }
      umma_commit(acc_full);  // always (see the big-tile kernel)
    }
  } else {
    // ---------------------------------------------------------------- decode
    // warp w: 16-input block w % J of code strip 2s + (w / J) % 2, K steps
    // ks = w / 2J (mod kSPar), J = blocks per K step
    const int blk = warp % T::kJobs;
    const int half = (warp / T::kJobs) % 2;
    const int ks0 = warp / kSJobs;
    const int g = OP8 ? dec_tile8(lane) : dec_tile(lane), c = lane & 3;
    const size_t row_bytes = (size_t)(p.out / 16) * 32 * K;
    // code strip of this warp: strip 2s + half, or (fused) strip s of gate
    // (half 0) or up (half 1)
    const int pg = p.fused ? half : pj;
    const uint8_t* cbase = reinterpret_cast<const uint8_t*>(gemm_expert_codes(p, e, pg)) +
                           (size_t)8 * (p.fused ? s : 2 * s + half) * 32 * K;
    const int n_my = (nks - ks0 + kSPar - 1) / kSPar;
    int off[8], off8[4];
#pragma unroll
    for (int idx = 0; idx < 8; idx++) {
      const int hf = idx >> 2, jh = (idx >> 1) & 1, jl = idx & 1;
      const int kr = c + 4 * jh;
      off[idx] = (g >> 2) * 1024 + hf * 4096 + kr * 128 + (((2 * (g & 3) + jl) ^ kr) << 4);
    }
#pragma unroll
    for (int c4 = 0; c4 < 4; c4++) {
      const int hf = c4 >> 1, kr = c + 4 * (c4 & 1);
      off8[c4] = hf * 2048 + kr * 128 + ((g ^ kr) << 4);
    }
    // a block of 16 inputs spans two 8-input groups; a code strip is one
    // (E4M3) or two (fp16) 1024-byte atoms wide
    const int job_off = OP8 ? blk * 4096 + half * 1024 : blk * 8192 + half * 2048;
    const uint32_t neg16 = opaque_u32(0xFFFF0000u);
    auto lane_codes = [&](int n) {
      const int ks = ks0 + n * kSPar;
      return reinterpret_cast<const uint16_t*>(cbase + (size_t)(ks * T::kJobs + blk) * row_bytes) +
             (g * 4 + c) * 4 * K;
    };
    constexpr int kL2Ahead = 4;
    auto prefetch_l2 = [&](int n) {
      if (n < n_my && lane * 128 < 8 * 32 * K) {
        const int ks = ks0 + n * kSPar;
        const uint8_t* a = cbase + (size_t)(ks * T::kJobs + blk) * row_bytes + lane * 128;
        asm volatile("prefetch.global.L2 [%0];" ::"l"(a));
      }
    };
    for (int n = 0; n < kL2Ahead; n++) prefetch_l2(n);
    const uint16_t* suh_e = (pg ? p.suh[1] : p.suh[0]) + (size_t)e * p.in + 16 * blk + c;
    uint32_t s2n[4];
    auto load_suh = [&](int n) {
      const int ks = ks0 + n * kSPar;
#pragma unroll
      for (int q = 0; q < 4; q++)  // format v2, FP8 operands: suh is on the activation side
        s2n[q] = p.had || OP8 ? 0x3C00u : __ldg(suh_e + ks * kKS + 4 * (q & 1) + 8 * (q >> 1));
    };
    LaneWords<K> nxt;
    if (n_my > 0) {
      load_suh(0);
      load_lane_words<K>(nxt, lane_codes(0));
    }
    int sw = ks0;
    uint32_t pw = 0;
    for (int n = 0; n < n_my; n++) {
      LaneWords<K> lw = nxt;
      if (n + 1 < n_my) load_lane_words<K>(nxt, lane_codes(n + 1));
      prefetch_l2(n + kL2Ahead);
      uint32_t s2[4];
#pragma unroll
      for (int q = 0; q < 4; q++) s2[q] = s2n[q] | (s2n[q] << 16);
      if (n + 1 < n_my) load_suh(n + 1);
      fetch_neighbour<K>(lw);
      if (!__all_sync(0xffffffffu, pipe_wait(&w_empty[sw], pw ^ 1, p, abort_flag))) break;
      if (OP8)
        decode_store8<K>(lw, p.mult, neg16, smem + sw * kSWStage + job_off, off8);
      else
        decode_store<K, FP8>(lw, p.mult, neg16, smem + sw * kSWStage + job_off, off, s2);
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&w_full[sw]);
      sw += kSPar;
      if (sw >= kSWStages) {
        sw -= kSWStages;
        pw ^= 1;
      }
    }

    // ------------------------------------------------------------- epilogue
    // warp w reads TMEM lanes 32 (w % 4) .. + 31, which hold tokens
    // 16 (w % 4) + lane, lane < 16 (M 64) or 32 (w % 4) + lane (M 128); it
    // takes output columns 64 (w / 4) .. + 63
    const bool live = epilogue_live(acc_full, p, abort_flag, abort_flag + 1, kSDec * 32);
    tc_fence_after();
    const int q4 = warp & 3, cg = warp >> 2;
    const bool lane_live = tm == 128 || lane < 16;
    const int n = (tm == 128 ? 32 : 16) * q4 + lane;  // token of this lane
    const uint32_t trow = tmem + ((uint32_t)(32 * q4) << 16);
    const uint16_t* svh = (pj ? p.svh[1] : p.svh[0]) + (size_t)e * p.out + kSN * s;
    if (live && p.fused) {
      // SwiGLU: this lane's token has gate output 128 s + j in column j and
      // up output 128 s + j in column 128 + j; warp (q4, cg) takes outputs
      // 32 cg .. 32 cg + 31 of the chunk and stores 32 fp16 h of its token
      const uint16_t* svg = p.svh[0] + (size_t)e * p.out + 128 * s;
      const uint16_t* svu = p.svh[1] + (size_t)e * p.out + 128 * s;
#pragma unroll
      for (int hc = 0; hc < 2; hc++) {
        const int c0 = 32 * cg + 16 * hc;
        float ag[16], au[16];
        tmem_ld16(trow + c0, ag);
        tmem_ld16(trow + 128 + c0, au);
        tmem_ld_wait(ag);
        tmem_ld_wait(au);
        if (lane_live && n < cnt) {
          const uint4 g0 = __ldg(reinterpret_cast<const uint4*>(svg + c0));
          const uint4 g1 = __ldg(reinterpret_cast<const uint4*>(svg + c0 + 8));
          const uint4 u0 = __ldg(reinterpret_cast<const uint4*>(svu + c0));
          const uint4 u1 = __ldg(reinterpret_cast<const uint4*>(svu + c0 + 8));
          const uint32_t gw[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
          const uint32_t uw[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
          const float sc = s_scale[n], hsc = __int_as_float(s_pid[n]);
          uint32_t hw[8];
#pragma unroll
          for (int j2 = 0; j2 < 8; j2++) {
            float hv[2];
#pragma unroll
            for (int b = 0; b < 2; b++) {
              const int j = 2 * j2 + b;
              const float sg = __half2float(__ushort_as_half((unsigned short)(b ? gw[j2] >> 16 : gw[j2] & 0xFFFFu)));
              const float su = __half2float(__ushort_as_half((unsigned short)(b ? uw[j2] >> 16 : uw[j2] & 0xFFFFu)));
              hv[b] = silu_f(ag[j] * sc * sg) * (au[j] * sc * su) * hsc;
            }
            hw[j2] = pack_h2(hv[0], hv[1]);
          }
          uint4* dst = reinterpret_cast<uint4*>(p.h_out + (size_t)(pos0 + n) * p.out + 128 * s + c0);
          dst[0] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
          dst[1] = make_uint4(hw[4], hw[5], hw[6], hw[7]);
        }
      }
    }
    if (live && p.had) {
      // Format v2: warps (q4, 2b) and (q4, 2b + 1) hold the two halves of the
      // 128-output block b for the same 32 TMEM lanes (tokens).  Both stage
      // their columns in shared memory (the weight ring is idle once the
      // accumulator is complete; [row][129] floats, conflict free both ways),
      // then each takes every other token row with lane l holding outputs
      // l + 32 j, rotates (j in registers, l by shuffles), scales and stores
      // 128 contiguous outputs of the row.
      const int blk = cg >> 1, hlf = cg & 1;
      float* xbuf = reinterpret_cast<float*>(smem) + (size_t)(2 * q4 + blk) * (32 * 129);
#pragma unroll
      for (int c = 0; c < 4; c++) {
        float a0[16];
        tmem_ld16(trow + 64 * cg + 16 * c, a0);
        tmem_ld_wait(a0);
#pragma unroll
        for (int i = 0; i < 16; i++) xbuf[lane * 129 + 64 * hlf + 16 * c + i] = a0[i];
      }
      named_bar_sync(1 + 2 * q4 + blk, 64);
      float svr[4];
#pragma unroll
      for (int j = 0; j < 4; j++)
        svr[j] = __half2float(__ushort_as_half(svh[128 * blk + lane + 32 * j]));
      const int rows = tm == 128 ? 32 : 16;
      for (int r = hlf; r < rows; r += 2) {
        float v[4];
#pragma unroll
        for (int j = 0; j < 4; j++) v[j] = xbuf[r * 129 + lane + 32 * j];
        wht_regs(v);
#pragma unroll
        for (int m = 1; m < 32; m <<= 1)
#pragma unroll
          for (int j = 0; j < 4; j++) v[j] = wht_lane(v[j], m, 0xffffffffu);
        const int nr = rows * q4 + r;
        if (nr < cnt) {
          const float sc = s_scale[nr];
          float* dst = p.gu_out ? p.gu_out + ((size_t)pj * p.n_pos + pos0 + nr) * p.out
                                : p.r_out + (size_t)s_pid[nr] * p.out;
#pragma unroll
          for (int j = 0; j < 4; j++) dst[kSN * s + 128 * blk + lane + 32 * j] = v[j] * sc * svr[j];
        }
      }
    }
    for (int c0 = p.had || p.fused || !live ? 64 * cg + 64 : 64 * cg; c0 < 64 * cg + 64; c0 += 16) {
      float a0[16];
      tmem_ld16(trow + c0, a0);
      tmem_ld_wait(a0);
      if (lane_live && n < cnt) {
        const uint4 sva = __ldg(reinterpret_cast<const uint4*>(svh + c0));
        const uint4 svb = __ldg(reinterpret_cast<const uint4*>(svh + c0 + 8));
        const uint32_t sw8[8] = {sva.x, sva.y, sva.z, sva.w, svb.x, svb.y, svb.z, svb.w};
        const float sc = s_scale[n];
        float v[16];
#pragma unroll
        for (int j = 0; j < 16; j++) {
          const uint32_t w2 = sw8[j >> 1];
          const float sv = __half2float(__ushort_as_half((unsigned short)(j & 1 ? w2 >> 16 : w2 & 0xFFFFu)));
          v[j] = a0[j] * sc * sv;
        }
        float* dst = !p.r_out ? p.gu_out + ((size_t)pj * p.n_pos + pos0 + n) * p.out
                              : p.r_out + (size_t)s_pid[n] * p.out;
        float4* d4 = reinterpret_cast<float4*>(dst + kSN * s + c0);
#pragma unroll
        for (int q = 0; q < 4; q++) d4[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kSDec) {
    mbar_drain(acc_full, 0, p.budget);  // every MMA issued has completed
    tc_fence_after();
    tmem_dealloc(tmem, kSN);
  }
}

// Row kernels: one warp per position row, 16-byte vector accesses; the first
// kRowCache chunks of 32 lanes x 8 (gather) or x 4 (swiglu) elements stay in
// registers between the max pass and the write pass, the rest are re-read.
constexpr int kRowWarps = 8;
constexpr int kRowCache = 16;

// Bound on |h| per expert for the fused SwiGLU epilogue: with |v| <= 4 (the
// codebook, E4M3 rule included) and the fp16 rounding of v * suh, |g_o| <=
// 8 max|suh_g| max|svh_g| |x|_1, likewise u, and |silu(g) u| <= |g| |u|, so
// |h| <= hb[e] |x|_1^2 with hb[e] = 64 max|suh_g| max|svh_g| max|suh_u|
// max|svh_u|.  CTAs 0 .. E-1: one expert each; the rest: |x_t|_1 of 8
// tokens each (one warp per token).
__global__ void __launch_bounds__(256) side_bound_kernel(const uint16_t* __restrict__ suh_g,
                                                         const uint16_t* __restrict__ suh_u,
                                                         const uint16_t* __restrict__ svh_g,
                                                         const uint16_t* __restrict__ svh_u,
                                                         int E, int H, int I,
                                                         const void* __restrict__ x, int x_bf16,
                                                         int T, float* __restrict__ hb,
                                                         float* __restrict__ l1) {
  pdl_wait();
  __shared__ float s_w[4][8];
  if ((int)blockIdx.x >= E) {
    const int t = (blockIdx.x - E) * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (t >= T) return;
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(x) + (size_t)t * H);
    float a = 0.0f;
    for (int v = lane; v < H / 8; v += 32) {
      float f[8];
      act8(src[v], x_bf16, f);
#pragma unroll
      for (int q = 0; q < 8; q++) a += fabsf(f[q]);
    }
    for (int off = 16; off > 0; off >>= 1) a += __shfl_xor_sync(0xffffffffu, a, off);
    if (lane == 0) l1[t] = a;
    return;
  }
  const int e = blockIdx.x;
  float m[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  auto fmax16 = [](float a, uint16_t b) { return fmaxf(a, fabsf(__half2float(__ushort_as_half(b)))); };
  for (int i = threadIdx.x; i < H; i += blockDim.x) {
    m[0] = fmax16(m[0], suh_g[(size_t)e * H + i]);
    m[1] = fmax16(m[1], suh_u[(size_t)e * H + i]);
  }
  for (int i = threadIdx.x; i < I; i += blockDim.x) {
    m[2] = fmax16(m[2], svh_g[(size_t)e * I + i]);
    m[3] = fmax16(m[3], svh_u[(size_t)e * I + i]);
  }
#pragma unroll
  for (int q = 0; q < 4; q++) {
    m[q] = warp_max(m[q]);
    if ((threadIdx.x & 31) == 0) s_w[q][threadIdx.x >> 5] = m[q];
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float r = 64.0f;
#pragma unroll
    for (int q = 0; q < 4; q++) {
      float a = 0.0f;
      for (int w = 0; w < (int)(blockDim.x >> 5); w++) a = fmaxf(a, s_w[q][w]);
      r *= a;
    }
    hb[e] = r;
  }
}

// Format v1 input pass: one warp per token.  Its row (bf16 or fp16) is read
// once, scaled to fp16 by the power of two that puts its amax in [2^14,
// 2^15), and written to the positions of the token's pairs that fall in the
// call's expert range (identical rows: the activation boxes of every segment
// the token is in); xinv[pos] = the inverse scale.  (One warp per position
// would read each token's row once per pair, and with the written rows
// streaming through L2 those reads come from HBM.)
__global__ void __launch_bounds__(kRowWarps * 32) gather_rows_kernel(
    const void* __restrict__ x, int x_bf16, int H, int k, int T,
    const int32_t* __restrict__ pair_pos, const int32_t* pos_lo, const int32_t* pos_hi,
    uint16_t* __restrict__ xg, float* __restrict__ xinv) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * kRowWarps + (threadIdx.x >> 5);
  if (t >= T) return;
  const int lo = *pos_lo, hi = *pos_hi;
  int my_pos = -1;  // lane j < k: position of pair t k + j, if in range
  if (lane < k) {
    const int ps = pair_pos[(size_t)t * k + lane];
    if (ps >= lo && ps < hi) my_pos = ps;
  }
  const unsigned used = __ballot_sync(0xffffffffu, my_pos >= 0);
  if (!used) return;  // none of this token's pairs is the call's
  const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(x) + (size_t)t * H);
  const int nv = H / 8;  // 16-byte vectors per row
  uint4 c[kRowCache];
  float am = 0.0f;
#pragma unroll
  for (int i = 0; i < kRowCache; i++) {
    const int v = i * 32 + lane;
    if (v < nv) {
      c[i] = src[v];
      float f[8];
      act8(c[i], x_bf16, f);
#pragma unroll
      for (int q = 0; q < 8; q++) am = fmaxf(am, fabsf(f[q]));
    }
  }
  for (int v = kRowCache * 32 + lane; v < nv; v += 32) {
    float f[8];
    act8(src[v], x_bf16, f);
#pragma unroll
    for (int q = 0; q < 8; q++) am = fmaxf(am, fabsf(f[q]));
  }
  am = warp_max(am);
  const int ex = fp16_scale_exp(am);
  const float sc = ldexpf(1.0f, ex);
  auto conv = [&](const uint4& r) {
    float f[8];
    act8(r, x_bf16, f);
    return make_uint4(pack_h2(f[0] * sc, f[1] * sc), pack_h2(f[2] * sc, f[3] * sc),
                      pack_h2(f[4] * sc, f[5] * sc), pack_h2(f[6] * sc, f[7] * sc));
  };
#pragma unroll
  for (int i = 0; i < kRowCache; i++)
    if (i * 32 + lane < nv) c[i] = conv(c[i]);
  for (unsigned m = used; m; m &= m - 1) {
    const int pos = __shfl_sync(0xffffffffu, my_pos, __ffs(m) - 1);
    uint4* dst = reinterpret_cast<uint4*>(xg + (size_t)pos * H);
#pragma unroll
    for (int i = 0; i < kRowCache; i++) {
      const int v = i * 32 + lane;
      if (v < nv) dst[v] = c[i];
    }
    for (int v = kRowCache * 32 + lane; v < nv; v += 32) dst[v] = conv(src[v]);
    if (lane == 0) xinv[pos] = ldexpf(1.0f, -ex);
  }
}

// Rows x * suh of gate and up for each position (gate rows at [pos], up rows
// at [P + pos]), for the layers whose suh cannot fold into the decoded
// weights: format v2 (ROT: each 128-input block rotated; the rotation sits
// between suh and the codes) and the FP8 operand mode (ACT8).  One warp per
// position; lane l holds inputs 8v .. 8v + 7 of vector v = 32 i + l, so a
// 128-block is 16 consecutive lanes (3 index bits in registers, 4 by
// shuffles; H is a multiple of 128, so both half-warps are active or idle
// together).
//   ACT8 = 0: fp16 rows with a power-of-two scale per row that also removes
//     the rotations' factor 128.  The scale comes from a bound instead of the
//     rotated values: an entry of a rotated block is at most the block's L1
//     norm, so the first pass needs no rotation (the power-of-two scale only
//     has to keep fp16 finite; it does not change the relative rounding of
//     normal fp16 values).
//   ACT8 = 1: E4M3 bytes q = E4M3(a / s), s = amax / 448 over the exact
//     (rotated) row, the row's scale s (times 2^-7 with the rotation).
template <int ROT, int ACT8>
__global__ void __launch_bounds__(kRowWarps * 32) gather_rows_split_kernel(
    const void* __restrict__ x, int x_bf16, int H, int k, int P, const int32_t* seg_pairs,
    const int32_t* pos_lo, const int32_t* pos_hi, const int32_t* ids,
    const uint16_t* __restrict__ suh_g, const uint16_t* __restrict__ suh_u,
    void* __restrict__ xg, float* __restrict__ xinv) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int pos = blockIdx.x * kRowWarps + (threadIdx.x >> 5);
  if (pos >= P || pos < *pos_lo || pos >= *pos_hi) return;  // outside the call's experts
  const int pr = seg_pairs[pos];
  const int t = pr / k, e = ids[pr];
  const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(x) + (size_t)t * H);
  const uint4* sg = reinterpret_cast<const uint4*>(suh_g + (size_t)e * H);
  const uint4* su = reinterpret_cast<const uint4*>(suh_u + (size_t)e * H);
  const int nv = H / 8;
  const unsigned hm = 0xFFFFu << (lane & 16);
  auto prods = [&](int v, float (&fg)[8], float (&fu)[8]) {
    float fx[8], a[8], b[8];
    act8(src[v], x_bf16, fx);
    act8(sg[v], 0, a);
    act8(su[v], 0, b);
#pragma unroll
    for (int q = 0; q < 8; q++) {
      fg[q] = fx[q] * a[q];
      fu[q] = fx[q] * b[q];
    }
  };
  auto rows = [&](int v, float (&fg)[8], float (&fu)[8]) {
    prods(v, fg, fu);
    if (ROT) {
      wht_regs(fg);
      wht_regs(fu);
#pragma unroll
      for (int m = 1; m < 16; m <<= 1)
#pragma unroll
        for (int q = 0; q < 8; q++) {
          fg[q] = wht_lane(fg[q], m, hm);
          fu[q] = wht_lane(fu[q], m, hm);
        }
    }
  };
  // pass 1: the largest magnitude (ACT8) or the largest block L1 norm
  float ag = 0.0f, au = 0.0f;
  for (int v = lane; v < nv; v += 32) {
    float fg[8], fu[8];
    if (ACT8) {
      rows(v, fg, fu);
#pragma unroll
      for (int q = 0; q < 8; q++) {
        ag = fmaxf(ag, fabsf(fg[q]));
        au = fmaxf(au, fabsf(fu[q]));
      }
    } else {
      prods(v, fg, fu);
      float lg = 0.0f, lu = 0.0f;
#pragma unroll
      for (int q = 0; q < 8; q++) {
        lg += fabsf(fg[q]);
        lu += fabsf(fu[q]);
      }
#pragma unroll
      for (int m = 1; m < 16; m <<= 1) {
        lg += __shfl_xor_sync(hm, lg, m);
        lu += __shfl_xor_sync(hm, lu, m);
      }
      ag = fmaxf(ag, lg);
      au = fmaxf(au, lu);
    }
  }
  ag = warp_max(ag);
  au = warp_max(au);
  const int hs = ROT ? kHadShift : 0;  // the unnormalized rotations' 128
  if (ACT8) {
    const float s_g = e4m3_row_scale(ag), s_u = e4m3_row_scale(au);
    const float r_g = s_g > 0.0f ? __frcp_rn(s_g) : 0.0f, r_u = s_u > 0.0f ? __frcp_rn(s_u) : 0.0f;
    uint2* dg = reinterpret_cast<uint2*>(static_cast<uint8_t*>(xg) + (size_t)pos * H);
    uint2* du = reinterpret_cast<uint2*>(static_cast<uint8_t*>(xg) + ((size_t)P + pos) * H);
    auto q8 = [](const float (&f)[8], float sc, float rc) {
      return make_uint2(e4m3_pair_of(f[0], f[1], sc, rc) | (e4m3_pair_of(f[2], f[3], sc, rc) << 16),
                        e4m3_pair_of(f[4], f[5], sc, rc) | (e4m3_pair_of(f[6], f[7], sc, rc) << 16));
    };
    for (int v = lane; v < nv; v += 32) {
      float fg[8], fu[8];
      rows(v, fg, fu);
      dg[v] = q8(fg, s_g, r_g);
      du[v] = q8(fu, s_u, r_u);
    }
    if (lane == 0) {
      xinv[pos] = ldexpf(s_g, -hs);
      xinv[(size_t)P + pos] = ldexpf(s_u, -hs);
    }
    return;
  }
  const int eg = fp16_scale_exp(ag), eu = fp16_scale_exp(au);
  const float scg = ldexpf(1.0f, eg), scu = ldexpf(1.0f, eu);
  uint4* dg = reinterpret_cast<uint4*>(static_cast<uint16_t*>(xg) + (size_t)pos * H);
  uint4* du = reinterpret_cast<uint4*>(static_cast<uint16_t*>(xg) + ((size_t)P + pos) * H);
  for (int v = lane; v < nv; v += 32) {
    float fg[8], fu[8];
    rows(v, fg, fu);
    dg[v] = make_uint4(pack_h2(fg[0] * scg, fg[1] * scg), pack_h2(fg[2] * scg, fg[3] * scg),
                       pack_h2(fg[4] * scg, fg[5] * scg), pack_h2(fg[6] * scg, fg[7] * scg));
    du[v] = make_uint4(pack_h2(fu[0] * scu, fu[1] * scu), pack_h2(fu[2] * scu, fu[3] * scu),
                       pack_h2(fu[4] * scu, fu[5] * scu), pack_h2(fu[6] * scu, fu[7] * scu));
  }
  if (lane == 0) {
    xinv[pos] = ldexpf(1.0f, -eg - hs);
    xinv[(size_t)P + pos] = ldexpf(1.0f, -eu - hs);
  }
}

// h = silu(g) * u per position row, the down projection's activation rows.
// Format v1 with fp16 operands: h itself (suh of down is applied on the
// weight side by the decoders), fp16 with a power-of-two row scale.  With
// the rotation (ROT, format v2) or FP8 operands (ACT8), h * suh_d of the
// position's expert (ROT: each 128-block rotated; lane l holds elements
// 4v .. 4v + 3 of v = 32 i + l: 2 index bits in registers, 5 by shuffles; I
// is a multiple of 128), the scale also removing the factor 128 of the
// rotations.  ACT8 stores E4M3 bytes q = E4M3(a / s), s = amax / 448, and
// the row scale s.
template <int ROT, int ACT8>
__global__ void __launch_bounds__(kRowWarps * 32) swiglu_rows_kernel(
    const float* __restrict__ gu, size_t n_pos, int I, const int32_t* seg_pairs,
    const int32_t* pos_lo, const int32_t* pos_hi, const int32_t* ids,
    const uint16_t* __restrict__ suh_d, void* __restrict__ hs, float* __restrict__ hinv) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const size_t pos = (size_t)blockIdx.x * kRowWarps + (threadIdx.x >> 5);
  if (pos >= n_pos || pos < (size_t)*pos_lo || pos >= (size_t)*pos_hi) return;
  const float4* gr = reinterpret_cast<const float4*>(gu + pos * I);
  const float4* ur = reinterpret_cast<const float4*>(gu + (n_pos + pos) * I);
  const int nv = I / 4;
  constexpr bool kSide = ROT || ACT8;
  const uint2* sd = kSide ? reinterpret_cast<const uint2*>(suh_d + (size_t)ids[seg_pairs[pos]] * I)
                          : nullptr;
  // times suh_d, then (ROT) rotated (every lane active: nv % 32 == 0)
  auto side = [&](float4& h, int v) {
    const uint2 sr = __ldg(sd + v);
    float w[4] = {h.x * __half2float(__ushort_as_half((unsigned short)(sr.x & 0xFFFFu))),
                  h.y * __half2float(__ushort_as_half((unsigned short)(sr.x >> 16))),
                  h.z * __half2float(__ushort_as_half((unsigned short)(sr.y & 0xFFFFu))),
                  h.w * __half2float(__ushort_as_half((unsigned short)(sr.y >> 16)))};
    if (ROT) {
      wht_regs(w);
#pragma unroll
      for (int m = 1; m < 32; m <<= 1)
#pragma unroll
        for (int q = 0; q < 4; q++) w[q] = wht_lane(w[q], m, 0xffffffffu);
    }
    h = make_float4(w[0], w[1], w[2], w[3]);
  };
  auto h4 = [&](int v) {
    const float4 g = __ldcs(gr + v), u = __ldcs(ur + v);
    float4 h = make_float4(silu_f(g.x) * u.x, silu_f(g.y) * u.y, silu_f(g.z) * u.z,
                           silu_f(g.w) * u.w);
    if (kSide) side(h, v);
    return h;
  };
  auto amax4 = [](float a, const float4& h) {
    return fmaxf(fmaxf(a, fabsf(h.x)), fmaxf(fmaxf(fabsf(h.y), fabsf(h.z)), fabsf(h.w)));
  };
  // the row's first chunks: every load issued before the first SiLU
  float4 c[kRowCache], cu[kRowCache];
  float am = 0.0f;
#pragma unroll
  for (int i = 0; i < kRowCache; i++) {
    const int v = i * 32 + lane;
    if (v < nv) {
      c[i] = __ldcs(gr + v);
      cu[i] = __ldcs(ur + v);
    }
  }
#pragma unroll
  for (int i = 0; i < kRowCache; i++) {
    const int v = i * 32 + lane;
    if (v < nv) {
      c[i] = make_float4(silu_f(c[i].x) * cu[i].x, silu_f(c[i].y) * cu[i].y,
                         silu_f(c[i].z) * cu[i].z, silu_f(c[i].w) * cu[i].w);
      if (kSide) side(c[i], v);
      am = amax4(am, c[i]);
    }
  }
  for (int v = kRowCache * 32 + lane; v < nv; v += 32) am = amax4(am, h4(v));
  am = warp_max(am);
  const int hsh = ROT ? kHadShift : 0;
  if (ACT8) {
    const float sc = e4m3_row_scale(am);
    const float rc = sc > 0.0f ? __frcp_rn(sc) : 0.0f;
    uint32_t* dst = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(hs) + pos * I);
    auto put = [&](int v, const float4& h) {
      dst[v] = e4m3_byte_of(h.x, sc, rc) | (e4m3_byte_of(h.y, sc, rc) << 8) |
               (e4m3_byte_of(h.z, sc, rc) << 16) | (e4m3_byte_of(h.w, sc, rc) << 24);
    };
#pragma unroll
    for (int i = 0; i < kRowCache; i++) {
      const int v = i * 32 + lane;
      if (v < nv) put(v, c[i]);
    }
    for (int v = kRowCache * 32 + lane; v < nv; v += 32) put(v, h4(v));
    if (lane == 0) hinv[pos] = ldexpf(sc, -hsh);
    return;
  }
  const int ex = fp16_scale_exp(am);
  const float sc = ldexpf(1.0f, ex);
  uint2* dst = reinterpret_cast<uint2*>(static_cast<uint16_t*>(hs) + pos * I);
  auto put = [&](int v, const float4& h) {
    dst[v] = make_uint2(pack_h2(h.x * sc, h.y * sc), pack_h2(h.z * sc, h.w * sc));
  };
#pragma unroll
  for (int i = 0; i < kRowCache; i++) {
    const int v = i * 32 + lane;
    if (v < nv) put(v, c[i]);
  }
  for (int v = kRowCache * 32 + lane; v < nv; v += 32) put(v, h4(v));
  if (lane == 0) hinv[pos] = ldexpf(1.0f, -ex - hsh);
}

// Token tiles per expert segment (one CTA, thread per expert): tiles of
// <= kBN positions in `tiles`; an expert's last tile (or its only one) goes
// to `tiles_s` instead when it holds <= kSM positions and use_small is set
// (the small-tile kernel).
// n_tiles[0] / n_tiles[1] receive the two counts.
__device__ int block_excl_scan(int v, int* s_warp, int* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int x = v;
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) s_warp[wid] = x;
  __syncthreads();
  if (wid == 0) {
    int u = lane < nw ? s_warp[lane] : 0;
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, u, off);
      if (lane >= off) u += y;
    }
    if (lane < nw) s_warp[lane] = u;
  }
  __syncthreads();
  const int r = (wid > 0 ? s_warp[wid - 1] : 0) + x - v;
  *total = s_warp[nw - 1];
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(1024) build_tiles_kernel(int E, const int32_t* seg_offsets,
                                                           int use_small, Shard sh, int32_t* tiles,
                                                           int32_t* tiles_s, int32_t* n_tiles) {
  pdl_wait();
  __shared__ int s_warp[32];
  const int e = threadIdx.x;
  // experts outside the call's range get no tiles
  const int cnt = e < E && e >= sh.e0 && e < sh.e1 ? seg_offsets[e + 1] - seg_offsets[e] : 0;
  const int nt = (cnt + kBN - 1) / kBN;
  const int last = nt > 0 ? cnt - (nt - 1) * kBN : 0;
  const int small = use_small && nt > 0 && last <= kSM ? 1 : 0;
  const int nbig = nt - small;
  int tot_b = 0, tot_s = 0;
  const int base_b = block_excl_scan(nbig, s_warp, &tot_b);
  const int base_s = block_excl_scan(small, s_warp, &tot_s);
  if (e < E) {
    const int off = seg_offsets[e];
    for (int j = 0; j < nbig; j++) {
      int32_t* t = tiles + (size_t)(base_b + j) * 4;
      t[0] = e;
      t[1] = off + j * kBN;
      t[2] = min(kBN, cnt - j * kBN);
      t[3] = 0;
    }
    if (small) {
      int32_t* t = tiles_s + (size_t)base_s * 4;
      t[0] = e;
      t[1] = off + nbig * kBN;
      t[2] = last;
      t[3] = 0;
    }
  }
  if (threadIdx.x == 0) {
    n_tiles[0] = tot_b;
    n_tiles[1] = tot_s;
  }
}

// Mixed widths: split the (tile, projection) work of the four launches (big
// and small tiles; gate/up and down) into one list per width.  Thread per
// (tile, projection p of 3).  Segments (in pairs): big gate/up 3 x 2mt, big
// down 3 x mt, small gate/up 3 x 2E, small down 3 x E; counts[kind * 6 +
// launch * 3 + width].  The order inside a list does not matter.
__global__ void __launch_bounds__(256) gemm_width_lists_kernel(
    const int32_t* __restrict__ n_tiles, const int32_t* __restrict__ tiles,
    const int32_t* __restrict__ tiles_s, const int32_t* __restrict__ kt, int mt, int E,
    int32_t* __restrict__ counts, int32_t* __restrict__ entries) {
  pdl_wait();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  const int small = i >= 3 * mt;
  const int j = small ? i - 3 * mt : i;
  const int t = j / 3, pg = j % 3;
  if (t >= (small ? n_tiles[1] : n_tiles[0]) || (small && t >= E)) return;
  const int e = (small ? tiles_s : tiles)[4 * t];
  const int w = kt[(size_t)e * 3 + pg] - 2;
  const int launch = pg == 2 ? 1 : 0;
  const int n = small ? E : mt;  // tiles of this kind at most
  const size_t seg = small ? (size_t)9 * mt + (launch ? (size_t)6 * E : 0)
                           : (launch ? (size_t)6 * mt : 0);
  const size_t cap = launch ? (size_t)n : (size_t)2 * n;
  const int slot = atomicAdd(&counts[small * 6 + launch * 3 + w], 1);
  int32_t* en = entries + (seg + (size_t)w * cap + slot) * 2;
  en[0] = t;
  en[1] = launch ? 0 : pg;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

// Row-major matrix [rows][cols] of fp16 (esize 2) or E4M3 bytes (esize 1) as
// a TMA source of boxes of 64 rows x 128 bytes, 128B swizzle.
bool make_tmap(CUtensorMap* m, const void* base, size_t rows, size_t cols, int esize) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * esize};
  cuuint32_t box[2] = {(cuuint32_t)(kRow / esize), 64};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, esize == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
            const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int K, int FP8, int OP8>
cudaError_t launch_gemm(const CUtensorMap& tm, const GemmParams& gp, int grid, cudaStream_t st) {
  using C = GCfg<K>;
  static bool init = false;
  auto kfn = gemm_kernel<K, FP8, OP8>;
  if (!init) {
    cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    init = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(OpT<OP8>::kThreads, 1, 1);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t err = cudaLaunchKernelEx(&cfg, kfn, tm, gp);
  note_launches(1);
  return err;
}

template <int K, int FP8, int OP8>
cudaError_t launch_gemm64(const CUtensorMap& tm, const GemmParams& gp, int grid, cudaStream_t st) {
  static bool init = false;
  auto kfn = gemm64_kernel<K, FP8, OP8>;
  if (!init) {
    cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, SCfg::kSmem);
    if (e != cudaSuccess) return e;
    init = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kSThreads, 1, 1);
  cfg.dynamicSmemBytes = SCfg::kSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t err = cudaLaunchKernelEx(&cfg, kfn, tm, gp);
  note_launches(1);
  return err;
}

// E4M3 operands (op8) exist only with the E4M3 rule (fp8).
cudaError_t dispatch_gemm64(int K, int fp8, int op8, const CUtensorMap& tm, const GemmParams& gp,
                            int grid, cudaStream_t st) {
  if (op8) {
    if (K == 2) return launch_gemm64<2, 1, 1>(tm, gp, grid, st);
    if (K == 3) return launch_gemm64<3, 1, 1>(tm, gp, grid, st);
    return launch_gemm64<4, 1, 1>(tm, gp, grid, st);
  }
  if (fp8) {
    if (K == 2) return launch_gemm64<2, 1, 0>(tm, gp, grid, st);
    if (K == 3) return launch_gemm64<3, 1, 0>(tm, gp, grid, st);
    return launch_gemm64<4, 1, 0>(tm, gp, grid, st);
  }
  if (K == 2) return launch_gemm64<2, 0, 0>(tm, gp, grid, st);
  if (K == 3) return launch_gemm64<3, 0, 0>(tm, gp, grid, st);
  return launch_gemm64<4, 0, 0>(tm, gp, grid, st);
}

cudaError_t dispatch_gemm(int K, int fp8, int op8, const CUtensorMap& tm, const GemmParams& gp,
                          int grid, cudaStream_t st) {
  if (op8) {
    if (K == 2) return launch_gemm<2, 1, 1>(tm, gp, grid, st);
    if (K == 3) return launch_gemm<3, 1, 1>(tm, gp, grid, st);
    return launch_gemm<4, 1, 1>(tm, gp, grid, st);
  }
  if (fp8) {
    if (K == 2) return launch_gemm<2, 1, 0>(tm, gp, grid, st);
    if (K == 3) return launch_gemm<3, 1, 0>(tm, gp, grid, st);
    return launch_gemm<4, 1, 0>(tm, gp, grid, st);
  }
  if (K == 2) return launch_gemm<2, 0, 0>(tm, gp, grid, st);
  if (K == 3) return launch_gemm<3, 0, 0>(tm, gp, grid, st);
  return launch_gemm<4, 0, 0>(tm, gp, grid, st);
}

size_t al(size_t b) { return (b + 255) & ~(size_t)255; }

// Test hook of the bounded waits (exl3_test_set_wait_fault): which gate/up
// tensor-core launch skips one K step's activation loads, and the clock
// budget of that launch's waits.
struct WaitFault {
  int kernel = 0;  // 0 none, 1 big-tile kernel, 2 small-tile kernel (gate/up launch)
  int ks = -1;
  long long budget = kWaitBudgetCycles;
};
WaitFault g_fault;

size_t max_tiles(int T, int E, int top_k) {
  const size_t P = (size_t)T * top_k;
  return (P + kBN - 1) / kBN + ((size_t)E < P ? (size_t)E : P);
}

struct GemmLayout {
  size_t xg, xinv, gu, hs, hinv, r, tiles, tiles_s, ntiles, counts, lists, hb, hl1, total;
};

// Format v2 and the FP8 operand mode keep separate gate and up activation
// rows (2P rows); FP8 rows are 1 byte per element.
GemmLayout gemm_layout(int T, int top_k, int E, int H, int I, int had, int act8) {
  GemmLayout g{};
  const size_t P = (size_t)T * top_k;
  const size_t xr = had || act8 ? 2 * P : P;
  size_t o = 0;
  g.xg = o; o += al(xr * H * (act8 ? 1 : 2));
  g.xinv = o; o += al(xr * 4);
  g.gu = o; o += al(2 * P * I * 4);
  g.hs = o; o += al(P * I * 2);
  g.hinv = o; o += al(P * 4);
  g.r = o; o += al(P * H * 4);
  g.tiles = o; o += al(max_tiles(T, E, top_k) * 16);
  g.tiles_s = o; o += al((size_t)E * 16);
  g.ntiles = o; o += al(16);
  g.counts = o; o += al(12 * 4);  // mixed widths: list lengths
  g.lists = o; o += al((size_t)18 * (max_tiles(T, E, top_k) + E) * 4);
  g.hb = o; o += al((size_t)E * 4);  // fused SwiGLU: per-expert bound on |h|
  g.hl1 = o; o += al((size_t)T * 4);  // and per-token |x|_1
  g.total = o;
  return g;
}

}  // namespace

size_t gemm_scratch_bytes(int T, int top_k, int E, int H, int I, int had, int act8) {
  return gemm_layout(T, top_k, E, H, I, had, act8).total;
}

cudaError_t launch_moe_gemm(const LayerView& L, const void* x, int x_bf16, int T, int top_k,
                            const RouteBuffers& rb, void* ws, const cudaEvent_t* ev, float** r_out,
                            Shard sh, cudaStream_t st) {
  auto rec = [&](int i) {
    if (ev && ev[i]) record_stage_event(ev[i], st);
  };
  const int a8 = L.act8;
  const bool split = L.had || a8;  // separate gate and up activation rows
  // SwiGLU in the gate/up epilogue: gate and up share the activation row
  // (format v1, fp16 operands) and one code width
  const bool fused = !split && !L.mixed;
  const int esize = a8 ? 1 : 2;
  const GemmLayout g = gemm_layout(T, top_k, L.E, L.H, L.I, L.had, a8);
  char* base = static_cast<char*>(ws);
  uint16_t* xg = reinterpret_cast<uint16_t*>(base + g.xg);
  float* xinv = reinterpret_cast<float*>(base + g.xinv);
  float* gu_buf = reinterpret_cast<float*>(base + g.gu);
  uint16_t* hs = reinterpret_cast<uint16_t*>(base + g.hs);
  float* hinv = reinterpret_cast<float*>(base + g.hinv);
  float* r = reinterpret_cast<float*>(base + g.r);
  int32_t* tiles = reinterpret_cast<int32_t*>(base + g.tiles);
  int32_t* tiles_s = reinterpret_cast<int32_t*>(base + g.tiles_s);
  int32_t* ntiles = reinterpret_cast<int32_t*>(base + g.ntiles);
  int32_t* lcounts = reinterpret_cast<int32_t*>(base + g.counts);
  int32_t* lists = reinterpret_cast<int32_t*>(base + g.lists);
  float* hb = reinterpret_cast<float*>(base + g.hb);
  float* hl1 = reinterpret_cast<float*>(base + g.hl1);
  *r_out = r;
  const int P = T * top_k;
  const int mt = (int)max_tiles(T, L.E, top_k);
  CUtensorMap tm_x, tm_h;
  if (!make_tmap(&tm_x, xg, (size_t)P * (split ? 2 : 1), (size_t)L.H, esize) ||
      !make_tmap(&tm_h, hs, (size_t)P, (size_t)L.I, esize))
    return cudaErrorInvalidValue;
  cudaError_t err;
  // grids: big tiles on 128-output strips, small tiles on 256-output chunks
  // (the small-tile kernel needs H and I to be multiples of 256; otherwise
  // every tile takes the big-tile kernel)
  const bool small_ok = L.H % kSN == 0 && L.I % kSN == 0;
  // positions of the call's experts: [seg_offsets[e0], seg_offsets[e1])
  const int32_t* pos_lo = rb.seg_offsets + sh.e0;
  const int32_t* pos_hi = rb.seg_offsets + sh.e1;
  if ((err = launch_pdl(build_tiles_kernel, dim3(1), dim3(1024), 0, st, L.E,
                        (const int32_t*)rb.seg_offsets, (int)small_ok, sh, tiles, tiles_s, ntiles)) !=
      cudaSuccess)
    return err;
  if (L.mixed) {
    if ((err = cudaMemsetAsync(lcounts, 0, 12 * sizeof(int32_t), st)) != cudaSuccess) return err;
    const int threads = 3 * (mt + L.E);
    err = launch_pdl(gemm_width_lists_kernel, dim3((unsigned)((threads + 255) / 256)), dim3(256), 0,
                     st, (const int32_t*)ntiles, (const int32_t*)tiles, (const int32_t*)tiles_s,
                     L.d_kt, mt, L.E, lcounts, lists);
    note_launches(1);
    if (err != cudaSuccess) return err;
  }
  // one launch of a kernel, or (mixed widths) one per width over its list;
  // kind 0 = big tiles, 1 = small tiles; launch 0 = gate/up, 1 = down
  auto run = [&](int kind, int launch, const CUtensorMap& tm, const GemmParams& gp, int grid,
                 int K) -> cudaError_t {
    auto one = [&](int k, const GemmParams& q) {
      return kind ? dispatch_gemm64(k, L.fp8, a8, tm, q, grid, st)
                  : dispatch_gemm(k, L.fp8, a8, tm, q, grid, st);
    };
    if (!L.mixed) return one(K, gp);
    const size_t n = kind ? (size_t)L.E : (size_t)mt;
    const size_t seg = kind ? (size_t)9 * mt + (launch ? (size_t)6 * L.E : 0)
                            : (launch ? (size_t)6 * mt : 0);
    const size_t cap = launch ? n : 2 * n;
    for (int w = 0; w < 3; w++) {
      if (!((L.wmask[launch] >> w) & 1)) continue;  // no expert has this width
      GemmParams q = gp;
      q.entries = lists + (seg + (size_t)w * cap) * 2;
      q.n_entries = lcounts + kind * 6 + launch * 3 + w;
      q.off = L.d_off;
      const cudaError_t e2 = one(w + 2, q);
      if (e2 != cudaSuccess) return e2;
    }
    return cudaSuccess;
  };
  const int row_blocks = (P + kRowWarps - 1) / kRowWarps;
  if (a8) {
    auto kfn = L.had ? gather_rows_split_kernel<1, 1> : gather_rows_split_kernel<0, 1>;
    err = launch_pdl(kfn, dim3(row_blocks), dim3(kRowWarps * 32), 0, st, x, x_bf16, L.H, top_k, P,
                     (const int32_t*)rb.seg_pairs, pos_lo, pos_hi, (const int32_t*)rb.ids,
                     L.suh[0], L.suh[1], (void*)xg, xinv);
  } else if (split) {
    err = launch_pdl(gather_rows_split_kernel<1, 0>, dim3(row_blocks), dim3(kRowWarps * 32), 0, st,
                     x, x_bf16, L.H, top_k, P, (const int32_t*)rb.seg_pairs, pos_lo, pos_hi,
                     (const int32_t*)rb.ids, L.suh[0], L.suh[1], (void*)xg, xinv);
  } else {
    if (fused) {
      err = launch_pdl(side_bound_kernel, dim3(L.E + (T + 7) / 8), dim3(256), 0, st, L.suh[0],
                       L.suh[1], L.svh[0], L.svh[1], L.E, L.H, L.I, x, x_bf16, T, hb, hl1);
      note_launches(1);
      if (err != cudaSuccess) return err;
    }
    err = launch_pdl(gather_rows_kernel, dim3((unsigned)((T + kRowWarps - 1) / kRowWarps)),
                     dim3(kRowWarps * 32), 0, st, x, x_bf16, L.H, top_k, T,
                     (const int32_t*)rb.pair_pos, pos_lo, pos_hi, xg, xinv);
  }
  note_launches(2);
  if (err != cudaSuccess) return err;
  rec(2);

  GemmParams gu{};
  gu.codes[0] = L.codes[0]; gu.codes[1] = L.codes[1];
  gu.stride[0] = L.code_stride[0]; gu.stride[1] = L.code_stride[1];
  gu.suh[0] = L.suh[0]; gu.suh[1] = L.suh[1];
  gu.svh[0] = L.svh[0]; gu.svh[1] = L.svh[1];
  gu.in = L.H; gu.out = L.I; gu.nproj = fused ? 1 : 2; gu.mult = L.mult;
  gu.tiles = tiles; gu.n_tiles = ntiles; gu.xinv = xinv; gu.n_pos = (size_t)P;
  gu.gu_out = fused ? nullptr : gu_buf;
  gu.fused = fused;
  gu.h_out = fused ? hs : nullptr;
  gu.hinv = hinv;
  gu.hb = hb;
  gu.l1 = hl1;
  gu.top_k = top_k;
  gu.seg_pairs = rb.seg_pairs;
  gu.status = rb.status;
  gu.budget = kWaitBudgetCycles;
  gu.fault_ks = -1;
  gu.had = L.had;
  gu.xrow_off = split ? P : 0;
  gu.proj0 = 0;
  const WaitFault wf = g_fault;
  auto with_fault = [&](GemmParams q, int kernel) {
    if (wf.kernel == kernel) {
      q.fault_ks = wf.ks;
      q.budget = wf.budget;
    }
    return q;
  };
  // without mixed widths gate and up share a width (one launch)
  if ((err = run(0, 0, tm_x, with_fault(gu, 1), mt * 2 * (L.I / 128), L.K[0])) != cudaSuccess)
    return err;
  if (small_ok) {
    GemmParams gs = with_fault(gu, 2);
    gs.tiles = tiles_s;
    gs.n_tiles = ntiles + 1;
    if ((err = run(1, 0, tm_x, gs, L.E * 2 * (L.I / kSN), L.K[0])) != cudaSuccess) return err;
  }
  rec(3);

  if (!fused) {
    auto kfn = L.had ? (a8 ? swiglu_rows_kernel<1, 1> : swiglu_rows_kernel<1, 0>)
                     : (a8 ? swiglu_rows_kernel<0, 1> : swiglu_rows_kernel<0, 0>);
    err = launch_pdl(kfn, dim3(row_blocks), dim3(kRowWarps * 32), 0, st, (const float*)gu_buf,
                     (size_t)P, L.I, (const int32_t*)rb.seg_pairs, pos_lo, pos_hi,
                     (const int32_t*)rb.ids, L.suh[2], (void*)hs, hinv);
    note_launches(1);
    if (err != cudaSuccess) return err;
  }
  rec(4);

  GemmParams dn{};
  dn.codes[0] = L.codes[2]; dn.stride[0] = L.code_stride[2];
  dn.suh[0] = L.suh[2]; dn.svh[0] = L.svh[2];
  dn.in = L.I; dn.out = L.H; dn.nproj = 1; dn.mult = L.mult;
  dn.tiles = tiles; dn.n_tiles = ntiles; dn.xinv = hinv; dn.r_out = r;
  dn.seg_pairs = rb.seg_pairs; dn.wts = rb.w; dn.status = rb.status;
  dn.budget = kWaitBudgetCycles;
  dn.fault_ks = -1;
  dn.had = L.had;
  dn.proj0 = 2;
  err = run(0, 1, tm_h, dn, mt * (L.H / 128), L.K[2]);
  if (err == cudaSuccess && small_ok) {
    GemmParams ds = dn;
    ds.tiles = tiles_s;
    ds.n_tiles = ntiles + 1;
    err = run(1, 1, tm_h, ds, L.E * (L.H / kSN), L.K[2]);
  }
  rec(5);
  return err;
}

}  // namespace exl3

namespace exl3 {
namespace {
// Rows of fp32 values to their E4M3 operand bytes and fp32 scales, with the
// device functions the activation passes use (one CTA per row).
__global__ void __launch_bounds__(256) quantize_rows_e4m3_kernel(const float* __restrict__ a, int n,
                                                                 uint8_t* __restrict__ q,
                                                                 float* __restrict__ s) {
  __shared__ float s_w[8];
  const float* row = a + (size_t)blockIdx.x * n;
  float am = 0.0f;
  for (int i = threadIdx.x; i < n; i += blockDim.x) am = fmaxf(am, fabsf(row[i]));
  am = warp_max(am);
  if ((threadIdx.x & 31) == 0) s_w[threadIdx.x >> 5] = am;
  __syncthreads();
  am = 0.0f;
  for (int w = 0; w < (int)(blockDim.x >> 5); w++) am = fmaxf(am, s_w[w]);
  const float sc = e4m3_row_scale(am);
  const float rc = sc > 0.0f ? __frcp_rn(sc) : 0.0f;
  // pairs of elements, as the activation passes take them (an odd last one alone)
  for (int i = 2 * threadIdx.x; i < n; i += 2 * blockDim.x) {
    if (i + 1 < n) {
      const uint32_t two = e4m3_pair_of(row[i], row[i + 1], sc, rc);
      q[(size_t)blockIdx.x * n + i] = (uint8_t)(two & 0xFFu);
      q[(size_t)blockIdx.x * n + i + 1] = (uint8_t)(two >> 8);
    } else {
      q[(size_t)blockIdx.x * n + i] = (uint8_t)e4m3_byte_of(row[i], sc, rc);
    }
  }
  if (threadIdx.x == 0) s[blockIdx.x] = sc;
}
}  // namespace
}  // namespace exl3

extern "C" exl3_status exl3_quantize_rows_e4m3(const float* a, int rows, int n, uint8_t* q,
                                               float* s, void* stream) {
  if (rows < 0 || n < 0) return EXL3_ERR_SHAPE;
  if (rows == 0 || n == 0) return EXL3_OK;
  if (!a || !q || !s) return EXL3_ERR_ARG;
  exl3::quantize_rows_e4m3_kernel<<<rows, 256, 0, static_cast<cudaStream_t>(stream)>>>(a, n, q, s);
  exl3::note_launches(1);
  return cudaGetLastError() == cudaSuccess ? EXL3_OK : EXL3_ERR_CUDA;
}

extern "C" exl3_status exl3_test_set_wait_fault(int kernel, int ks, long long budget_cycles) {
  if (kernel == 0) {
    exl3::g_fault = exl3::WaitFault{};
    return EXL3_OK;
  }
  if (kernel < 1 || kernel > 2 || ks < 0 || budget_cycles < 100000 ||
      budget_cycles > exl3::kWaitBudgetCycles)
    return EXL3_ERR_ARG;
  exl3::g_fault.kernel = kernel;
  exl3::g_fault.ks = ks;
  exl3::g_fault.budget = budget_cycles;
  return EXL3_OK;
}
