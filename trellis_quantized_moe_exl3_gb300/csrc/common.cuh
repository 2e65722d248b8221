// Device helpers shared by the kernels of the EXL3 MoE library (sm_103a).
//
// Format v1 (the library's reading of the pages; "GLM-5.3-Flash EXL3 (~2.1
// bpw, SM70 tile order)" intro, "GLM-5.3-Flash · exlr8 (K2/K3/K4)" intro,
// Loading and Calibration):
//   * one 16x16 tile = 16*K little-endian uint16 words = a circular bit string
//     of 256*K bits, least significant bit of word 0 first;
//   * weight t's 16-bit state is the window of 16 bits starting at bit t*K;
//   * mcg codebook: x = state * mult (mod 2^32), m = (x & 0x8FFF8FFF) ^
//     0x3B603B60, whose 16-bit halves are two fp16 numbers a (low) and b (high);
//     the weight is fp16(a + b), optionally rounded to FP8 E4M3 (nearest even,
//     saturating) before the side vectors;
//   * tile order gb300_v1: weight t = 64c + 8r0 + 4hf + j sits at output row
//     r0 + 8(j&1) and input column c + 4(j>>1) + 8hf.
// Lane c (0..3) of an MMA quad owns bits [64cK, 64(c+1)K) of a tile, i.e. the
// 8K bytes at byte offset 8Kc, plus the first 16-K bits of lane c+1 (mod 4).
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace exl3 {

constexpr uint32_t kMcgMask = 0x8FFF8FFFu;
constexpr uint32_t kMcgXor = 0x3B603B60u;

// ---------------------------------------------------------------- routing exp
// exp for the routing softmax, defined for bit-exact agreement with any other
// implementation of the same rule: inputs below -86 (and -inf, NaN) give 0;
// n = rint(x*log2(e)); Cody-Waite reduction with the Cephes two-part ln2
// (0.693359375, -2.12194440e-4) by fma; degree-7 Taylor polynomial with fp32
// coefficients 1/n! in Horner form by fma; exact scaling by 2^n (n >= -124).
__device__ __forceinline__ float exp_route(float x) {
  if (!(x >= -86.0f)) return 0.0f;
  const float t = __fmul_rn(x, 0x1.715476p+0f);
  const float n = rintf(t);
  float r = __fmaf_rn(-n, 0x1.63p-1f, x);
  r = __fmaf_rn(-n, -0x1.bd0106p-13f, r);
  float p = 0x1.a01a02p-13f;            // 1/5040
  p = __fmaf_rn(p, r, 0x1.6c16c2p-10f);  // 1/720
  p = __fmaf_rn(p, r, 0x1.111112p-7f);   // 1/120
  p = __fmaf_rn(p, r, 0x1.555556p-5f);   // 1/24
  p = __fmaf_rn(p, r, 0x1.555556p-3f);   // 1/6
  p = __fmaf_rn(p, r, 0.5f);
  p = __fmaf_rn(p, r, 1.0f);
  p = __fmaf_rn(p, r, 1.0f);
  const int ni = (int)n;
  return __fmul_rn(p, __int_as_float((ni + 127) << 23));
}

// ---------------------------------------------------------------- trellis
// Number of 32-bit words a quad lane owns (8K bytes) plus one word of its
// right neighbour for the window overlap.
template <int K>
struct LaneWords {
  static constexpr int kOwn = 2 * K;
  uint32_t w[2 * K + 1];
};

// 32-bit window of the lane stream starting at bit o (o compile-time after
// unrolling); bits beyond the stream read as 0.
template <int K>
__device__ __forceinline__ uint32_t lane_window32(const LaneWords<K>& lw, int o) {
  const int wi = o >> 5;
  const int sh = o & 31;
  const uint32_t lo = lw.w[wi];
  const uint32_t hi = (wi + 1 < 2 * K + 1) ? lw.w[wi + 1] : 0u;
  return sh == 0 ? lo : __funnelshift_r(lo, hi, sh);
}

// An opaque register copy of a constant, so that a multiply by it stays an
// integer multiply-add (FMA pipe) instead of being rewritten as shifts.
__device__ __forceinline__ uint32_t opaque_u32(uint32_t v) {
  uint32_t r;
  asm("mov.b32 %0, %1;" : "=r"(r) : "r"(v));
  return r;
}

// The codebook's mask-xor, (x & 0x8FFF8FFF) ^ 0x3B603B60, as ONE three-input
// logic operation.  A LOP3 takes a single immediate, so with both constants
// as immediates the compiler splits it into two logic operations: one more
// ALU-pipe instruction per decoded weight, on the pipe that bounds the decode.
// The constants therefore come in registers (mcg_consts(), taken once per
// decode routine).
struct McgConsts {
  uint32_t mask, xr;
};
__device__ __forceinline__ McgConsts mcg_consts() {
  return McgConsts{opaque_u32(kMcgMask), opaque_u32(kMcgXor)};
}
__device__ __forceinline__ uint32_t mcg_maskxor(uint32_t x, const McgConsts& c) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(r) : "r"(x), "r"(c.mask), "r"(c.xr));
  return r;
}

// State of lane-local weight u (0..63): bits [uK, uK+16) of the lane stream.
// u is a compile-time constant after unrolling, so this is one funnel shift
// (or plain shift) and one mask.
template <int K>
__device__ __forceinline__ uint32_t lane_state(const LaneWords<K>& lw, int u) {
  const int o = u * K;
  const int wi = o >> 5;
  const int sh = o & 31;
  uint32_t v;
  if (sh == 0)
    v = lw.w[wi];
  else if (sh <= 16)
    v = lw.w[wi] >> sh;
  else
    v = __funnelshift_r(lw.w[wi], lw.w[wi + 1], sh);
  return v & 0xFFFFu;
}

// mcg codebook before the final add: the two fp16 halves {a (low), b (high)}.
__device__ __forceinline__ uint32_t mcg_halves(uint32_t s, uint32_t mult, const McgConsts& c) {
  return mcg_maskxor(s * mult, c);
}

// {a, b} halves of lane-local weight u.  For K = 2 and 4 the 16 bits above a
// weight's state are exactly the state of weight u + 16/K, so instead of
// masking the window to 16 bits the hash of the whole 32-bit window is taken
// and corrected: (s + 2^16 g) * M - ((g * M) << 16) = s * M (mod 2^32), where
// the low 16 bits of g * M are those of the next window's hash.  This trades
// two ALU-pipe operations (shift, mask) for one FMA-pipe multiply-add.  For
// K = 3 the window is masked.
template <int K>
__device__ __forceinline__ uint32_t lane_halves(const LaneWords<K>& lw, int u, uint32_t mult,
                                                uint32_t neg_shift16, const McgConsts& c) {
  if constexpr (K == 2 || K == 4) {
    constexpr int step = 16 / K;
    const uint32_t xa = lane_window32<K>(lw, u * K) * mult;
    const uint32_t xb = lane_window32<K>(lw, (u + step) * K) * mult;
    const uint32_t x = xb * neg_shift16 + xa;
    return mcg_maskxor(x, c);
  } else {
    return mcg_halves(lane_state<K>(lw, u), mult, c);
  }
}

// fp16 RNE of a + b for two weights at once: {a0,b0},{a1,b1} -> {v0,v1}.
__device__ __forceinline__ uint32_t sum_halves2(uint32_t m0, uint32_t m1) {
  const uint32_t lo = __byte_perm(m0, m1, 0x5410);  // {a0, a1}
  const uint32_t hi = __byte_perm(m0, m1, 0x7632);  // {b0, b1}
  __half2 r = __hadd2(*reinterpret_cast<const __half2*>(&lo),
                      *reinterpret_cast<const __half2*>(&hi));
  return *reinterpret_cast<uint32_t*>(&r);
}

// E4M3 rule on two fp16 values: round to FP8 E4M3 (RNE, satfinite) and back;
// every E4M3 value is exact in fp16.
__device__ __forceinline__ uint32_t e4m3_round2(uint32_t v2) {
  uint16_t f8;
  uint32_t back;
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(f8) : "r"(v2));
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(back) : "h"(f8));
  return back;
}

// The E4M3 rule on two fp16 values, kept as the two E4M3 bytes (low byte =
// the low fp16 value): the weight operand of the FP8 tensor-core path.
__device__ __forceinline__ uint32_t e4m3_bytes2(uint32_t v2) {
  uint16_t f8;
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(f8) : "r"(v2));
  return f8;
}

// Two fp32 values to E4M3 (RNE, satfinite) bytes: lo -> low byte, hi -> high byte.
__device__ __forceinline__ uint32_t e4m3_pack2(float lo, float hi) {
  uint16_t f8;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(f8) : "f"(hi), "f"(lo));
  return f8;
}

// Per-row E4M3 activation operand (the FP8 x FP8 product's activations):
// s = amax / 448 and q = E4M3_RNE_sat(a / s), both divisions IEEE fp32 (the
// precision in which the quantised code is decided); an all-zero row has
// s = 0 and q = 0.
__device__ __forceinline__ float e4m3_row_scale(float amax) {
  return amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 0.0f;
}

// E4M3 byte of a / s for one element, with r = 1 / s (correctly rounded,
// taken once per row).  p = a * r is within 2.5 fp32 ulps of the correctly
// rounded quotient Q = fp32(a / s) (r and the product each round once), so Q
// lies between the values 4 ulps below and above |p|.  E4M3 rounding is
// monotonic: when both of those round to the same byte, Q does too, and that
// byte is the decision an IEEE division would give.  Only a quotient within
// a few ulps of an E4M3 rounding boundary takes the IEEE division.
// (kept out of line so that the common path does not carry the division)
static __device__ __noinline__ uint32_t e4m3_byte_div(float a, float s) {
  return e4m3_pack2(fabsf(__fdiv_rn(a, s)), 0.0f) & 0xFFu;
}
__device__ __forceinline__ uint32_t e4m3_byte_of(float a, float s, float r) {
  if (!(s > 0.0f)) return 0u;
  const uint32_t m = __float_as_uint(a * r) & 0x7FFFFFFFu;
  const uint32_t two = e4m3_pack2(__uint_as_float(m > 4u ? m - 4u : 0u), __uint_as_float(m + 4u));
  uint32_t b = two & 0xFFu;
  if (__builtin_expect(b != (two >> 8), 0)) b = e4m3_byte_div(a, s);
  return b | (a < 0.0f ? 0x80u : 0u);
}

// Two elements at once (low byte = a0), the same decisions, cheaper: when
// |p| >= 2^-6 (E4M3's normal range, where every rounding boundary is a float
// whose 20 low mantissa bits are 0x80000) and p lies more than 5 ulps from
// such a float, no boundary separates p from fp32(a / s) (2.5 ulps away at
// most), so p itself is converted, two per instruction.  Any other element
// (a quotient near a boundary, a small or zero one) takes e4m3_byte_of; rows
// with many small elements (products such as h) do better with
// e4m3_byte_of throughout.
__device__ __forceinline__ bool e4m3_clear(float p) {
  const uint32_t m = __float_as_uint(p) & 0x7FFFFFFFu;
  return m >= 0x3C800000u && ((m & 0xFFFFFu) - 0x7FFFBu) > 10u;
}
__device__ __forceinline__ uint32_t e4m3_pair_of(float a0, float a1, float s, float r) {
  const float p0 = a0 * r, p1 = a1 * r;
  if (__builtin_expect(s > 0.0f && e4m3_clear(p0) && e4m3_clear(p1), 1))
    return e4m3_pack2(p0, p1);
  return e4m3_byte_of(a0, s, r) | (e4m3_byte_of(a1, s, r) << 8);
}

// The same element as a float (every E4M3 value is exact in fp16 and fp32).
__device__ __forceinline__ float e4m3_value(float a, float s, float r) {
  uint32_t back;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(back) : "h"((uint16_t)e4m3_byte_of(a, s, r)));
  return __half2float(__ushort_as_half((unsigned short)(back & 0xFFFFu)));
}

// Load a quad lane's 8K bytes from global memory (read once: no L1 allocate)
// and fetch the neighbour's first word with a shuffle inside the quad.
template <int K>
__device__ __forceinline__ void load_lane_words(LaneWords<K>& lw, const uint16_t* tile_lane) {
  if constexpr (K == 2) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(tile_lane));
    lw.w[0] = v.x; lw.w[1] = v.y; lw.w[2] = v.z; lw.w[3] = v.w;
  } else if constexpr (K == 3) {
#pragma unroll
    for (int q = 0; q < 3; q++) {
      uint2 v;
      asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];"
                   : "=r"(v.x), "=r"(v.y) : "l"(tile_lane + 4 * q));
      lw.w[2 * q] = v.x; lw.w[2 * q + 1] = v.y;
    }
  } else {
#pragma unroll
    for (int q = 0; q < 2; q++) {
      uint4 v;
      asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                   : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(tile_lane + 8 * q));
      lw.w[4 * q] = v.x; lw.w[4 * q + 1] = v.y; lw.w[4 * q + 2] = v.z; lw.w[4 * q + 3] = v.w;
    }
  }
}

// Neighbour word: lane c of a quad takes lane (c+1) mod 4's first word.
template <int K>
__device__ __forceinline__ void fetch_neighbour(LaneWords<K>& lw) {
  const int lane = threadIdx.x & 31;
  lw.w[2 * K] = __shfl_sync(0xffffffffu, lw.w[0], (lane & ~3) | ((lane + 1) & 3));
}

// ---------------------------------------------------------------- MMA
// D += A * B, m16n8k16, fp16 operands, fp32 accumulate (legacy warp MMA).
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                              uint32_t a2, uint32_t a3, uint32_t b0,
                                              uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ---------------------------------------------------------------- PDL
// Kernels of the forward chain are launched with programmatic dependent
// launch: a kernel may become resident while its stream predecessor drains,
// and must wait here before it touches memory the predecessor reads or writes.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---------------------------------------------------------------- Hadamard
// Format v2 rotation ("GLM-5.3-Flash · exlr8 (K2/K3/K4)", Calibration: a
// 128x128 Hadamard matrix is a format primitive): v . H over each 128-block,
// H the Sylvester matrix with entries (-1)^popcount(i & j).  It is applied
// unnormalized on both sides of a projection, so the product carries a factor
// 128 that a 2^-7 in the activation scale removes exactly.  The 7 index bits
// of a block are split between registers and lanes; a stage maps (a, b) to
// (a + b, a - b) over one index bit, and stages commute.
constexpr int kHadShift = 7;  // log2 of the block size

template <int N>
__device__ __forceinline__ void wht_regs(float (&v)[N]) {
#pragma unroll
  for (int h = 1; h < N; h <<= 1)
#pragma unroll
    for (int i = 0; i < N; i++)
      if (!(i & h)) {
        const float a = v[i], b = v[i + h];
        v[i] = a + b;
        v[i + h] = a - b;
      }
}

// One stage over lane bit m (partner lane ^ m, both inside `mask`): the lane
// with the bit clear keeps v + o, its partner o - v, both as one fma with a
// sign of +-1 (exact product, one rounding: the same result as the add).
__device__ __forceinline__ float wht_lane(float v, int m, unsigned mask) {
  const float o = __shfl_xor_sync(mask, v, m);
  return fmaf((threadIdx.x & m) ? -1.0f : 1.0f, v, o);
}

// ---------------------------------------------------------------- misc
__device__ __forceinline__ float load_act(const void* x, int is_bf16, size_t idx) {
  const uint16_t b = reinterpret_cast<const uint16_t*>(x)[idx];
  if (is_bf16) return __uint_as_float((uint32_t)b << 16);
  return __half2float(__ushort_as_half(b));
}

// Power-of-two exponent that maps amax into [2^14, 2^15), for fp16 operands.
__device__ __forceinline__ int fp16_scale_exp(float amax) {
  if (!(amax > 0.0f) || !isfinite(amax)) return 0;
  int e = ilogbf(amax);
  int s = 14 - e;
  return s < -100 ? -100 : (s > 100 ? 100 : s);
}

// SiLU with the fast exponential and division (relative error ~1e-6, far
// below the fp16 rounding of every consumer).
__device__ __forceinline__ float silu_f(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

}  // namespace exl3
