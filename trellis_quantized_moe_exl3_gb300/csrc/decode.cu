// Dense decode of one projection of one expert: codes -> fp16 [in][out].
// The check path for the format (page "GLM-5.3 Flash EXL3 for 2x DGX Sparks",
// section Cold prefill (E3): outputs compared with the dense LinearEXL3
// reference).  Bit-exact by construction: the fp16 sum a + b is one RNE add
// of an exact sum, the E4M3 rule is one hardware cvt (RNE, satfinite), the
// side vectors are two fp32 RNE multiplies and one fp16 RNE conversion.
//
// One warp decodes the 8 consecutive tiles (i, 8jg .. 8jg+7): quad g takes
// tile 8jg+g and lane c of the quad its 8K-byte quarter.
#include "common.cuh"
#include "internal.h"

namespace exl3 {

namespace {

template <int K, int FP8>
__global__ void __launch_bounds__(256) decode_dense_kernel(const uint16_t* __restrict__ codes,
                                                           int in, int out, uint32_t mult,
                                                           const uint16_t* __restrict__ suh,
                                                           const uint16_t* __restrict__ svh,
                                                           int apply_side,
                                                           uint16_t* __restrict__ dst) {
  const int ngroups = out / 128;
  const int nblk = in / 16;
  const int gw = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (gw >= nblk * ngroups) return;  // warp-uniform
  const int i = gw / ngroups, jg = gw % ngroups;
  const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
  const uint16_t* chunk = codes + ((size_t)i * (out / 16) + (size_t)jg * 8) * 16 * K;
  LaneWords<K> lw;
  load_lane_words<K>(lw, chunk + lane * 4 * K);
  fetch_neighbour<K>(lw);
  const int tj = jg * 8 + g;
  const uint32_t neg16 = opaque_u32(0xFFFF0000u);
  const McgConsts mc = mcg_consts();
#pragma unroll
  for (int u = 0; u < 64; u += 2) {
    const uint32_t m0 = lane_halves<K>(lw, u, mult, neg16, mc);
    const uint32_t m1 = lane_halves<K>(lw, u + 1, mult, neg16, mc);
    uint32_t v2 = sum_halves2(m0, m1);
    if (FP8) v2 = e4m3_round2(v2);
#pragma unroll
    for (int h = 0; h < 2; h++) {
      const int uu = u + h;
      const int r0 = uu >> 3, hf = (uu >> 2) & 1, j = uu & 3;
      const int row = r0 + 8 * (j & 1);
      const int col = c + 4 * (j >> 1) + 8 * hf;
      const int o = 16 * tj + row, q = 16 * i + col;
      uint16_t bits = (uint16_t)(h ? (v2 >> 16) : (v2 & 0xFFFFu));
      if (apply_side) {
        float f = __fmul_rn(__half2float(__ushort_as_half(bits)), __half2float(__ushort_as_half(suh[q])));
        f = __fmul_rn(f, __half2float(__ushort_as_half(svh[o])));
        bits = __half_as_ushort(__float2half_rn(f));
      }
      dst[(size_t)q * out + o] = bits;
    }
  }
}

template <int K>
cudaError_t launch_k(const LayerView& L, int expert, int proj, int apply_side, uint16_t* out,
                     cudaStream_t st) {
  const int in = proj == 2 ? L.I : L.H;
  const int outf = proj == 2 ? L.H : L.I;
  const uint16_t* codes = L.codes[proj] + layer_code_offset(L, expert, proj);
  const uint16_t* suh = L.suh[proj] + (size_t)expert * in;
  const uint16_t* svh = L.svh[proj] + (size_t)expert * outf;
  const int warps = (in / 16) * (outf / 128);
  const int blocks = (warps + 7) / 8;
  if (L.fp8)
    decode_dense_kernel<K, 1><<<blocks, 256, 0, st>>>(codes, in, outf, L.mult, suh, svh,
                                                      apply_side, out);
  else
    decode_dense_kernel<K, 0><<<blocks, 256, 0, st>>>(codes, in, outf, L.mult, suh, svh,
                                                      apply_side, out);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_dense(const LayerView& L, int expert, int proj, int apply_side,
                                uint16_t* out, cudaStream_t st) {
  switch (layer_width(L, expert, proj)) {
    case 2: return launch_k<2>(L, expert, proj, apply_side, out, st);
    case 3: return launch_k<3>(L, expert, proj, apply_side, out, st);
    default: return launch_k<4>(L, expert, proj, apply_side, out, st);
  }
}

}  // namespace exl3
