// Grouped GEMM path for prefill-sized steps on the 5th-generation tensor
// cores (tcgen05 + TMEM + TMA), with the trellis decoded into shared memory.
//
// Page "GLM-5.3 Flash EXL3 for 2x DGX Sparks", section Cold prefill (E3):
// three GPU-driven launches per MoE layer (gather; gate/up + SwiGLU; down +
// scatter) built from device-side segment tables.  Page "GLM-5.3-Flash ·
// exlr8 (K2/K3/K4)", Widths: with the E4M3 codebook, prefill runs on the
// tensor cores.
//
// One CTA = (token tile of <= 256 positions of one expert, 128-output strip).
// D[o][n] = sum_i W[i][o] x[n][i] with A = decoded weights (M = 128 outputs,
// MN-major in shared memory) and B = activation rows (N = tokens, K-major,
// loaded by TMA with 128-byte swizzle); fp16 operands, fp32 accumulators in
// TMEM (gate and up side by side for the first launch).
//   warps 0-7  decode: each takes one 16-input block of the 64-input K step
//              (gate/up: 2 projections x 4 blocks; down: 4 blocks, two K steps
//              in flight), streams its code rows with cp.async, sums the
//              codebook halves into fp16 (E4M3 rule if set), applies suh and
//              stores 16-byte chunks into the swizzled A stage;
//   warp 8     TMA producer of the B stages, and TMEM allocator;
//   warp 9     one thread issues tcgen05.mma and commits stage releases.
// The epilogue (warps 0-7) reads TMEM: gate/up -> h = silu(g) * u (fp32);
// down -> router weight * svh * acc into the pair's own row (no atomics).
#include <cuda.h>

#include "common.cuh"
#include "internal.h"
#include "pipeline.cuh"
#include "umma.cuh"

namespace exl3 {

namespace {

constexpr int kBN = 256;   // max tokens per tile (MMA N)
constexpr int kKS = 64;    // inputs per K step
constexpr int kDec = 8;    // decoder warps
constexpr int kThreads = (kDec + 2) * 32;
constexpr int kCodeStages = 4;
constexpr int kBStages = 3;
constexpr int kAProj = 128 * kKS * 2;   // 16 KB: one projection's A stage
constexpr int kBStage = kBN * kKS * 2;  // 32 KB

template <int K, int NPROJ>
struct GCfg {
  static constexpr int kJobs = NPROJ * 4;          // decode jobs per K step
  static constexpr int kPar = kDec / kJobs;        // K steps decoded in parallel
  static constexpr int kAStages = 2 * kPar;
  static constexpr int kAStage = NPROJ * kAProj;
  static constexpr int kCodeChunk = 8 * 32 * K;
  static constexpr int kOffB = kAStages * kAStage;
  static constexpr int kOffCode = kOffB + kBStages * kBStage;
  static constexpr int kOffBar = kOffCode + kDec * kCodeStages * kCodeChunk;
  static constexpr int kNumBars = 2 * kAStages + 2 * kBStages + 1;
  static constexpr int kSmem = kOffBar + kNumBars * 8 + 16 + 1024;  // + alignment slack
  static constexpr int kTmemCols = NPROJ * kBN;
};

struct GemmParams {
  const uint16_t* codes[2];
  size_t stride[2];         // uint16 words per expert
  const uint16_t* suh[2];   // [E][in]
  const uint16_t* svh[2];   // [E][out]
  int in, out;
  uint32_t mult;
  const int32_t* tiles;     // [t][4] {expert, pos0, count, 0}
  const int32_t* n_tiles;
  const float* xinv;        // [pos] scale of the B rows
  float* h_out;             // gate/up: [pos][out]
  float* r_out;             // down: [pair id][out]
  const int32_t* seg_pairs;
  const float* wts;
  int32_t* status;
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

template <int K>
__device__ __forceinline__ void lds_words(LaneWords<K>& lw, const uint8_t* p) {
#pragma unroll
  for (int q = 0; q < 2 * K; q += 2) {
    const uint2 v = *reinterpret_cast<const uint2*>(p + 4 * q);
    lw.w[q] = v.x;
    lw.w[q + 1] = v.y;
  }
}

// Decode this lane's 64 weights of one tile and store them into the MN-major
// A stage of one projection: lane (g, c) holds outputs 16g..16g+15 (rows of
// the strip) for inputs c, c+4, c+8, c+12 of block `blk`.
template <int K, int FP8>
__device__ __forceinline__ void decode_store(const LaneWords<K>& lw, uint32_t mult, uint8_t* a_proj,
                                             int blk, int g, int c, const uint16_t* suh_blk) {
  const uint32_t neg16 = opaque_u32(0xFFFF0000u);
  const int am = g >> 2;
  const int ch0 = 2 * (g & 3);
#pragma unroll
  for (int hf = 0; hf < 2; hf++) {
#pragma unroll
    for (int jh = 0; jh < 2; jh++) {
      const int i = c + 4 * jh + 8 * hf;
      const int k = 16 * blk + i;
      const uint16_t sb = __ldg(suh_blk + i);
      const uint32_t s2 = (uint32_t)sb | ((uint32_t)sb << 16);
#pragma unroll
      for (int jl = 0; jl < 2; jl++) {
        uint32_t v[4];
#pragma unroll
        for (int pp = 0; pp < 4; pp++) {
          const int u0 = 16 * pp + 4 * hf + 2 * jh + jl;
          const uint32_t m0 = lane_halves<K>(lw, u0, mult, neg16);
          const uint32_t m1 = lane_halves<K>(lw, u0 + 8, mult, neg16);
          uint32_t v2 = sum_halves2(m0, m1);
          if (FP8) v2 = e4m3_round2(v2);
          __half2 h = __hmul2(*reinterpret_cast<const __half2*>(&v2),
                              *reinterpret_cast<const __half2*>(&s2));
          v[pp] = *reinterpret_cast<uint32_t*>(&h);
        }
        const int off = am * 1024 + (k >> 3) * 2048 + (k & 7) * 128 + (((ch0 + jl) ^ (k & 7)) << 4);
        *reinterpret_cast<uint4*>(a_proj + off) = make_uint4(v[0], v[1], v[2], v[3]);
      }
    }
  }
}

template <int K, int FP8, int NPROJ>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmap_b, GemmParams p) {
  using C = GCfg<K, NPROJ>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~(uintptr_t)1023);
  const int strips = p.out / 128;
  const int tile = blockIdx.x / strips, s = blockIdx.x % strips;
  if (tile >= p.n_tiles[0]) return;
  const int e = p.tiles[4 * tile], pos0 = p.tiles[4 * tile + 1], cnt = p.tiles[4 * tile + 2];
  const int n_mma = ((cnt + 15) / 16) * 16;
  const int nbox = (n_mma + 63) / 64;
  const int nks = p.in / kKS;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* a_full = bars;
  uint64_t* a_empty = a_full + C::kAStages;
  uint64_t* b_full = a_empty + C::kAStages;
  uint64_t* b_empty = b_full + kBStages;
  uint64_t* acc_full = b_empty + kBStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kAStages; i++) {
      mbar_init(&a_full[i], C::kJobs);
      mbar_init(&a_empty[i], 1);
    }
    for (int i = 0; i < kBStages; i++) {
      mbar_init(&b_full[i], 1);
      mbar_init(&b_empty[i], 1);
    }
    mbar_init(acc_full, 1);
    fence_mbar_init();
  }
  if (warp == kDec) tmem_alloc(tmem_slot, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kDec) {
    // ---------------------------------------------------------------- TMA
    if (lane == 0) {
      for (int ks = 0; ks < nks; ks++) {
        const int sb = ks % kBStages;
        mbar_wait_or_abort(&b_empty[sb], ((ks / kBStages) & 1) ^ 1, p.status);
        mbar_arrive_expect_tx(&b_full[sb], nbox * 64 * kKS * 2);
        uint8_t* dst = smem + C::kOffB + sb * kBStage;
        for (int j = 0; j < nbox; j++)
          tma_load_2d(dst + j * 64 * kKS * 2, &tmap_b, ks * kKS, pos0 + 64 * j, &b_full[sb]);
      }
      // the last loads were consumed by the MMA thread unless it gave up:
      // wait (bounded) for them before the CTA may exit
      for (int ks = nks - kBStages < 0 ? 0 : nks - kBStages; ks < nks; ks++)
        mbar_wait_or_abort(&b_full[ks % kBStages], (ks / kBStages) & 1, p.status);
    }
  } else if (warp == kDec + 1) {
    // ---------------------------------------------------------------- MMA
    if (lane == 0) {
      const uint32_t idesc = umma_idesc_f16(128, n_mma, 1, 0);
      for (int ks = 0; ks < nks; ks++) {
        const int sa = ks % C::kAStages, sb = ks % kBStages;
        mbar_wait_or_abort(&a_full[sa], (ks / C::kAStages) & 1, p.status);
        mbar_wait_or_abort(&b_full[sb], (ks / kBStages) & 1, p.status);
        tc_fence_after();
        const uint32_t a_base = smem_u32(smem + sa * C::kAStage);
        const uint32_t b_base = smem_u32(smem + C::kOffB + sb * kBStage);
#pragma unroll
        for (int kk = 0; kk < kKS / 16; kk++) {
          const uint64_t bdesc = umma_desc(b_base + kk * 32, 16, 1024);
#pragma unroll
          for (int pj = 0; pj < NPROJ; pj++) {
            const uint64_t adesc = umma_desc(a_base + pj * kAProj + kk * 4096, 1024, 2048);
            umma_f16(tmem + pj * kBN, adesc, bdesc, idesc, (ks > 0 || kk > 0) ? 1u : 0u);
          }
        }
        umma_commit(&a_empty[sa]);
        umma_commit(&b_empty[sb]);
      }
      umma_commit(acc_full);
    }
  } else {
    // ---------------------------------------------------------------- decode
    const int job = warp % C::kJobs;
    const int pj = job / 4, blk = job % 4;
    const int ks0 = warp / C::kJobs;
    const int g = lane >> 2, c = lane & 3;
    uint8_t* ring = smem + C::kOffCode + warp * kCodeStages * C::kCodeChunk;
    const size_t row_bytes = (size_t)(p.out / 16) * 32 * K;
    const uint8_t* cbase = reinterpret_cast<const uint8_t*>(p.codes[pj] + p.stride[pj] * e) +
                           (size_t)8 * s * 32 * K;
    const int n_my = (nks - ks0 + C::kPar - 1) / C::kPar;
    auto issue = [&](int n) {
      const int ks = ks0 + n * C::kPar;
      const uint8_t* src = cbase + (size_t)(ks * 4 + blk) * row_bytes;
      uint8_t* dst = ring + (n % kCodeStages) * C::kCodeChunk;
#pragma unroll
      for (int q = 0; q < (C::kCodeChunk + 511) / 512; q++)
        if (q * 512 + lane * 16 < C::kCodeChunk) cp_async16(dst + q * 512 + lane * 16, src + q * 512 + lane * 16);
    };
#pragma unroll
    for (int n = 0; n < kCodeStages - 1; n++) {
      if (n < n_my) issue(n);
      cp_async_commit();
    }
    const uint16_t* suh_e = p.suh[pj] + (size_t)e * p.in;
    for (int n = 0; n < n_my; n++) {
      const int ks = ks0 + n * C::kPar;
      const int sa = ks % C::kAStages;
      if (n + kCodeStages - 1 < n_my) issue(n + kCodeStages - 1);
      cp_async_commit();
      cp_async_wait<kCodeStages - 1>();
      __syncwarp();
      LaneWords<K> lw;
      lds_words<K>(lw, ring + (n % kCodeStages) * C::kCodeChunk + lane * 8 * K);
      fetch_neighbour<K>(lw);
      mbar_wait_or_abort(&a_empty[sa], ((ks / C::kAStages) & 1) ^ 1, p.status);
      decode_store<K, FP8>(lw, p.mult, smem + sa * C::kAStage + pj * kAProj, blk, g, c,
                           suh_e + ks * kKS + 16 * blk);
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&a_full[sa]);
    }
    cp_async_wait<0>();

    // ------------------------------------------------------------- epilogue
    mbar_wait_or_abort(acc_full, 0, p.status);
    tc_fence_after();
    const int q4 = warp & 3, half = warp >> 2;
    const int o = 128 * s + 32 * q4 + lane;
    const uint32_t trow = tmem + ((uint32_t)(32 * q4) << 16);
    const float sv0 = __half2float(__ushort_as_half(p.svh[0][(size_t)e * p.out + o]));
    const float sv1 = NPROJ == 2 ? __half2float(__ushort_as_half(p.svh[1][(size_t)e * p.out + o])) : 0.f;
    for (int c0 = half * (kBN / 2); c0 < (half + 1) * (kBN / 2) && c0 < cnt; c0 += 16) {
      float a0[16];
      tmem_ld16(trow + c0, a0);
      if constexpr (NPROJ == 2) {
        float a1[16];
        tmem_ld16(trow + kBN + c0, a1);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; i++) {
          const int n = c0 + i;
          if (n < cnt) {
            const int pos = pos0 + n;
            const float xi = p.xinv[pos];
            const float G = a0[i] * xi * sv0, U = a1[i] * xi * sv1;
            p.h_out[(size_t)pos * p.out + o] = silu_f(G) * U;
          }
        }
      } else {
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; i++) {
          const int n = c0 + i;
          if (n < cnt) {
            const int pos = pos0 + n;
            const int pid = p.seg_pairs[pos];
            p.r_out[(size_t)pid * p.out + o] = a0[i] * p.xinv[pos] * sv0 * p.wts[pid];
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kDec) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// Activation rows in position order, fp16 with a power-of-two scale per row
// chosen from its max |x| (undone in the epilogue).
__global__ void __launch_bounds__(256) gather_rows_kernel(const void* __restrict__ x, int x_bf16,
                                                          int H, int k, const int32_t* seg_pairs,
                                                          uint16_t* __restrict__ xg,
                                                          float* __restrict__ xinv) {
  __shared__ float s_w[32];
  const int pos = blockIdx.x;
  const int t = seg_pairs[pos] / k;
  float am = 0.0f;
  for (int i = threadIdx.x; i < H; i += blockDim.x) am = fmaxf(am, fabsf(load_act(x, x_bf16, (size_t)t * H + i)));
  for (int off = 16; off > 0; off >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, off));
  if ((threadIdx.x & 31) == 0) s_w[threadIdx.x >> 5] = am;
  __syncthreads();
  am = 0.0f;
  for (int w = 0; w < (int)(blockDim.x >> 5); w++) am = fmaxf(am, s_w[w]);
  const int ex = fp16_scale_exp(am);
  const float sc = ldexpf(1.0f, ex);
  uint16_t* dst = xg + (size_t)pos * H;
  for (int i = threadIdx.x; i < H; i += blockDim.x)
    dst[i] = __half_as_ushort(__float2half_rn(load_act(x, x_bf16, (size_t)t * H + i) * sc));
  if (threadIdx.x == 0) xinv[pos] = ldexpf(1.0f, -ex);
}

// h rows as fp16 with a power-of-two row scale (suh of down is applied on
// the weight side by the decoder, like suh of gate and up).
__global__ void __launch_bounds__(256) rowscale_kernel(const float* __restrict__ h, int I,
                                                       uint16_t* __restrict__ hs,
                                                       float* __restrict__ hinv) {
  __shared__ float s_w[32];
  const int pos = blockIdx.x;
  const float* hr = h + (size_t)pos * I;
  float am = 0.0f;
  for (int i = threadIdx.x; i < I; i += blockDim.x) am = fmaxf(am, fabsf(hr[i]));
  for (int off = 16; off > 0; off >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, off));
  if ((threadIdx.x & 31) == 0) s_w[threadIdx.x >> 5] = am;
  __syncthreads();
  am = 0.0f;
  for (int w = 0; w < (int)(blockDim.x >> 5); w++) am = fmaxf(am, s_w[w]);
  const int ex = fp16_scale_exp(am);
  const float sc = ldexpf(1.0f, ex);
  uint16_t* dst = hs + (size_t)pos * I;
  for (int i = threadIdx.x; i < I; i += blockDim.x)
    dst[i] = __half_as_ushort(__float2half_rn(hr[i] * sc));
  if (threadIdx.x == 0) hinv[pos] = ldexpf(1.0f, -ex);
}

// Token tiles of <= kBN positions per expert segment (one CTA, thread per expert).
__global__ void __launch_bounds__(1024) build_tiles_kernel(int E, const int32_t* seg_offsets,
                                                           int32_t* tiles, int32_t* n_tiles) {
  __shared__ int s_warp[32];
  const int e = threadIdx.x;
  const int cnt = e < E ? seg_offsets[e + 1] - seg_offsets[e] : 0;
  const int nt = (cnt + kBN - 1) / kBN;
  // block exclusive scan of nt
  const int lane = e & 31, wid = e >> 5, nw = blockDim.x >> 5;
  int x = nt;
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) s_warp[wid] = x;
  __syncthreads();
  if (wid == 0) {
    int v = lane < nw ? s_warp[lane] : 0;
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, v, off);
      if (lane >= off) v += y;
    }
    if (lane < nw) s_warp[lane] = v;
  }
  __syncthreads();
  const int base = (wid > 0 ? s_warp[wid - 1] : 0) + x - nt;
  if (e < E) {
    const int off = seg_offsets[e];
    for (int j = 0; j < nt; j++) {
      int32_t* t = tiles + (size_t)(base + j) * 4;
      t[0] = e;
      t[1] = off + j * kBN;
      t[2] = min(kBN, cnt - j * kBN);
      t[3] = 0;
    }
  }
  if (threadIdx.x == 0) n_tiles[0] = s_warp[nw - 1];
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

// Row-major fp16 matrix [rows][cols] as a TMA source of 64 x 64 boxes, 128B swizzle.
bool make_tmap(CUtensorMap* m, const void* base, size_t rows, size_t cols) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {64, 64};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int K, int FP8, int NPROJ>
cudaError_t launch_gemm(const CUtensorMap& tm, const GemmParams& gp, int grid, cudaStream_t st) {
  using C = GCfg<K, NPROJ>;
  static bool init = false;
  auto kfn = gemm_kernel<K, FP8, NPROJ>;
  if (!init) {
    cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    init = true;
  }
  kfn<<<grid, kThreads, C::kSmem, st>>>(tm, gp);
  note_launches(1);
  return cudaGetLastError();
}

template <int NPROJ>
cudaError_t dispatch_gemm(int K, int fp8, const CUtensorMap& tm, const GemmParams& gp, int grid,
                          cudaStream_t st) {
  if (fp8) {
    if (K == 2) return launch_gemm<2, 1, NPROJ>(tm, gp, grid, st);
    if (K == 3) return launch_gemm<3, 1, NPROJ>(tm, gp, grid, st);
    return launch_gemm<4, 1, NPROJ>(tm, gp, grid, st);
  }
  if (K == 2) return launch_gemm<2, 0, NPROJ>(tm, gp, grid, st);
  if (K == 3) return launch_gemm<3, 0, NPROJ>(tm, gp, grid, st);
  return launch_gemm<4, 0, NPROJ>(tm, gp, grid, st);
}

size_t al(size_t b) { return (b + 255) & ~(size_t)255; }

size_t max_tiles(int T, int E, int top_k) {
  const size_t P = (size_t)T * top_k;
  return (P + kBN - 1) / kBN + ((size_t)E < P ? (size_t)E : P);
}

struct GemmLayout {
  size_t xg, xinv, h, hs, hinv, r, tiles, ntiles, total;
};

GemmLayout gemm_layout(int T, int top_k, int E, int H, int I) {
  GemmLayout g{};
  const size_t P = (size_t)T * top_k;
  size_t o = 0;
  g.xg = o; o += al(P * H * 2);
  g.xinv = o; o += al(P * 4);
  g.h = o; o += al(P * I * 4);
  g.hs = o; o += al(P * I * 2);
  g.hinv = o; o += al(P * 4);
  g.r = o; o += al(P * H * 4);
  g.tiles = o; o += al(max_tiles(T, E, top_k) * 16);
  g.ntiles = o; o += al(16);
  g.total = o;
  return g;
}

}  // namespace

size_t gemm_scratch_bytes(int T, int top_k, int E, int H, int I) {
  return gemm_layout(T, top_k, E, H, I).total;
}

cudaError_t launch_moe_gemm(const LayerView& L, const void* x, int x_bf16, int T, int top_k,
                            const RouteBuffers& rb, void* ws, const cudaEvent_t* ev, float** r_out,
                            cudaStream_t st) {
  auto rec = [&](int i) {
    if (ev && ev[i]) record_stage_event(ev[i], st);
  };
  const GemmLayout g = gemm_layout(T, top_k, L.E, L.H, L.I);
  char* base = static_cast<char*>(ws);
  uint16_t* xg = reinterpret_cast<uint16_t*>(base + g.xg);
  float* xinv = reinterpret_cast<float*>(base + g.xinv);
  float* h = reinterpret_cast<float*>(base + g.h);
  uint16_t* hs = reinterpret_cast<uint16_t*>(base + g.hs);
  float* hinv = reinterpret_cast<float*>(base + g.hinv);
  float* r = reinterpret_cast<float*>(base + g.r);
  int32_t* tiles = reinterpret_cast<int32_t*>(base + g.tiles);
  int32_t* ntiles = reinterpret_cast<int32_t*>(base + g.ntiles);
  *r_out = r;
  const int P = T * top_k;
  const int mt = (int)max_tiles(T, L.E, top_k);
  CUtensorMap tm_x, tm_h;
  if (!make_tmap(&tm_x, xg, (size_t)P, (size_t)L.H) || !make_tmap(&tm_h, hs, (size_t)P, (size_t)L.I))
    return cudaErrorInvalidValue;
  cudaError_t err;
  build_tiles_kernel<<<1, 1024, 0, st>>>(L.E, rb.seg_offsets, tiles, ntiles);
  gather_rows_kernel<<<P, 256, 0, st>>>(x, x_bf16, L.H, top_k, rb.seg_pairs, xg, xinv);
  note_launches(2);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  rec(2);

  GemmParams gu{};
  gu.codes[0] = L.codes[0]; gu.codes[1] = L.codes[1];
  gu.stride[0] = L.code_stride[0]; gu.stride[1] = L.code_stride[1];
  gu.suh[0] = L.suh[0]; gu.suh[1] = L.suh[1];
  gu.svh[0] = L.svh[0]; gu.svh[1] = L.svh[1];
  gu.in = L.H; gu.out = L.I; gu.mult = L.mult;
  gu.tiles = tiles; gu.n_tiles = ntiles; gu.xinv = xinv; gu.h_out = h; gu.status = rb.status;
  if ((err = dispatch_gemm<2>(L.K[0], L.fp8, tm_x, gu, mt * (L.I / 128), st)) != cudaSuccess)
    return err;
  rec(3);

  rowscale_kernel<<<P, 256, 0, st>>>(h, L.I, hs, hinv);
  note_launches(1);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  rec(4);

  GemmParams dn{};
  dn.codes[0] = L.codes[2]; dn.stride[0] = L.code_stride[2];
  dn.suh[0] = L.suh[2]; dn.svh[0] = L.svh[2];
  dn.in = L.I; dn.out = L.H; dn.mult = L.mult;
  dn.tiles = tiles; dn.n_tiles = ntiles; dn.xinv = hinv; dn.r_out = r;
  dn.seg_pairs = rb.seg_pairs; dn.wts = rb.w; dn.status = rb.status;
  err = dispatch_gemm<1>(L.K[2], L.fp8, tm_h, dn, mt * (L.H / 128), st);
  rec(5);
  return err;
}

}  // namespace exl3
