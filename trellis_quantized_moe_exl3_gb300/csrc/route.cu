// Top-k routing and device-side segment tables.
//
// Page "GLM-5.3-Flash · exlr8 (K2/K3/K4)", intro: 288 routed experts with
// top-8 routing.  Page "GLM-5.3 Flash EXL3 for 2x DGX Sparks", section Cold
// prefill (E3): the expert launches are built from device-side segment
// tables, with no per-expert launches and no host sync.
//
// Rules: experts by descending fp32 logit, ties to the lower index, NaN as
// -inf; w_j = e_j / sum_j e_j (fp32, summed in j order) with e_j =
// exp_route(l_j - l_max), the difference taken as 0 when l_j == l_max.
// seg_offsets[e] counts pairs with expert < e; seg_pairs lists pair ids
// t*k + j expert-major and ascending inside an expert (a stable counting
// sort: per-chunk counts, a scan over (expert, chunk), a scatter by rank).
//
// A layer whose shared expert is trellis-coded (page "GLM-5.3-Flash · exlr8
// (K2/K3/K4)", Loading: the shared expert is stored as expert 288, after the
// routed ones) routes it as one more pair per token: pair t*(k+1) + k has
// expert E (the logits' width) and weight 1, so the tables cover E + 1
// experts and the expert kernels treat it like any other segment.
#include "common.cuh"
#include "internal.h"

namespace exl3 {

namespace {

// Order-preserving unsigned key of a logit: a larger logit has a larger key,
// NaN counts as -inf and -0 as +0 (they compare equal as floats), and every
// key is above 0, which stands for "no candidate".
__device__ __forceinline__ uint32_t logit_key(float f) {
  if (isnan(f)) f = -INFINITY;
  if (f == 0.0f) f = 0.0f;
  const uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_logit(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// One warp selects the top-k of one token.  MAXPL = logits held per lane
// (lane l holds experts l, l + 32, ...).  Round j: each lane offers its best
// expert not yet taken (its lowest index among equal keys), one warp max over
// the keys and one warp min over the indices offering that key pick expert j.
template <int MAXPL>
__device__ __forceinline__ void warp_topk(const float* __restrict__ lrow, int E, int k,
                                          int* my_id, float* my_w) {
  const int lane = threadIdx.x & 31;
  uint32_t key[MAXPL];
#pragma unroll
  for (int i = 0; i < MAXPL; i++) {
    const int e = lane + 32 * i;
    key[i] = e < E ? logit_key(lrow[e]) : 0u;  // 0: never offered
  }
  uint32_t kmax = 0, mine_k = 0;
  int mine_e = 0;
  for (int j = 0; j < k; j++) {
    uint32_t bk = 0;
    int bi = 0;
#pragma unroll
    for (int i = 0; i < MAXPL; i++)
      if (key[i] > bk) {
        bk = key[i];
        bi = i;
      }
    const uint32_t m = __reduce_max_sync(0xffffffffu, bk);
    const int be = __reduce_min_sync(0xffffffffu, bk == m ? lane + 32 * bi : 0x7fffffff);
    if ((be & 31) == lane) {
#pragma unroll
      for (int i = 0; i < MAXPL; i++)
        if (i == (be >> 5)) key[i] = 0u;  // taken
    }
    if (lane == j) {
      mine_e = be;
      mine_k = m;
    }
    if (j == 0) kmax = m;
  }
  // softmax over the k selected, in j order
  const float lmax = key_logit(kmax), mine_l = key_logit(mine_k);
  float ex = 0.0f;
  if (lane < k) {
    const float d = (mine_l == lmax) ? 0.0f : __fsub_rn(mine_l, lmax);
    ex = exp_route(d);
  }
  float exs[kMaxTopK];
#pragma unroll
  for (int j = 0; j < kMaxTopK; j++) exs[j] = __shfl_sync(0xffffffffu, ex, j);
  float sum = 0.0f;
#pragma unroll
  for (int j = 0; j < kMaxTopK; j++)
    if (j < k) sum = __fadd_rn(sum, exs[j]);
  *my_id = mine_e;
  *my_w = (lane < k) ? __fdiv_rn(ex, sum) : 0.0f;
}

// Block-wide exclusive scan of one int per thread (blockDim.x <= 1024).
__device__ int block_exclusive_scan(int v, int* smem_warp, int* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int nw = (blockDim.x + 31) >> 5;
  int x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) smem_warp[wid] = x;
  __syncthreads();
  if (wid == 0) {
    int s = lane < nw ? smem_warp[lane] : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, s, off);
      if (lane >= off) s += y;
    }
    if (lane < nw) smem_warp[lane] = s;  // inclusive warp totals
  }
  __syncthreads();
  const int base = wid > 0 ? smem_warp[wid - 1] : 0;
  const int res = base + x - v;
  if (total) *total = smem_warp[nw - 1];
  __syncthreads();
  return res;
}

// Token groups of one expert: kGroup consecutive positions of its segment.
__device__ __forceinline__ void write_groups(const RouteBuffers& rb, int e, int off, int cnt,
                                             int goff) {
  rb.group_off[e] = goff;
  for (int j = 0; j * kGroup < cnt; j++) {
    int32_t* gr = rb.groups + (size_t)(goff + j) * 4;
    gr[0] = e;
    gr[1] = off + j * kGroup;
    gr[2] = min(kGroup, cnt - j * kGroup);
    gr[3] = 0;
  }
}

// Per-chunk stage: top-k of kRouteChunk tokens, local stable ranks and
// per-expert counts.  With `fused` (single chunk) it also finishes the
// tables: offsets, active list and scatter.  E: logits per token (routed
// experts); sh = 1 appends the shared pair (expert E, weight 1) to each token,
// so pairs are t * (k + sh) + j and the tables cover E + sh experts.
template <int MAXPL>
__global__ void __launch_bounds__(1024) route_chunk_kernel(const float* __restrict__ logits, int T,
                                                           int E, int k, int sh, RouteBuffers rb,
                                                           int fused) {
  pdl_wait();
  // routing is the first kernel of a call: it clears the device status word
  // (no kernel that may set a bit runs before it or beside it)
  if (blockIdx.x == 0 && threadIdx.x == 0) *rb.status = 0;
  static_assert(kRouteChunk <= 64, "one bit per token of a chunk");
  __shared__ int s_ids[kRouteChunk * (kMaxTopK + 1)];
  __shared__ int s_cnt[kMaxExperts];
  __shared__ unsigned long long s_tok[kMaxExperts];  // bit tl: token tl has the expert
  __shared__ int s_warp[32];
  const int chunk = blockIdx.x;
  const int t0 = chunk * kRouteChunk;
  const int nt = min(kRouteChunk, T - t0);
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int kp = k + sh, Et = E + sh;  // pairs per token, experts in the tables

  for (int e = threadIdx.x; e < Et; e += blockDim.x) s_tok[e] = 0ull;
  for (int tl = wid; tl < nt; tl += nw) {
    const int t = t0 + tl;
    int id;
    float wt;
    warp_topk<MAXPL>(logits + (size_t)t * E, E, k, &id, &wt);
    if (lane < k) {
      rb.ids[(size_t)t * kp + lane] = id;
      rb.w[(size_t)t * kp + lane] = wt;
      s_ids[tl * kp + lane] = id;
    } else if (lane < kp) {  // the shared expert
      rb.ids[(size_t)t * kp + lane] = E;
      rb.w[(size_t)t * kp + lane] = 1.0f;
      s_ids[tl * kp + lane] = E;
    }
  }
  __syncthreads();
  // stable local ranks: the rank of pair (tl, j) is the number of earlier
  // tokens of the chunk routed to the same expert (the k experts of a token
  // are distinct), read off the expert's token mask
  const int np = nt * kp;
  for (int pl = threadIdx.x; pl < np; pl += blockDim.x)
    atomicOr(&s_tok[s_ids[pl]], 1ull << (pl / kp));
  __syncthreads();
  auto rank_of = [&](int pl) {
    return __popcll(s_tok[s_ids[pl]] & ((1ull << (pl / kp)) - 1ull));
  };
  for (int e = threadIdx.x; e < Et; e += blockDim.x) s_cnt[e] = __popcll(s_tok[e]);
  if (!fused) {
    for (int pl = threadIdx.x; pl < np; pl += blockDim.x) rb.rank[(size_t)t0 * kp + pl] = rank_of(pl);
    for (int e = threadIdx.x; e < Et; e += blockDim.x)
      rb.chunk_counts[(size_t)chunk * Et + e] = s_cnt[e];
    return;
  }
  __syncthreads();
  // fused: offsets = exclusive scan of the counts, active list, scatter
  int total = 0, n_act = 0, n_grp = 0;
  const int cnt = threadIdx.x < Et ? s_cnt[threadIdx.x] : 0;
  const int off = block_exclusive_scan(cnt, s_warp, &total);
  const int aidx = block_exclusive_scan(cnt > 0 ? 1 : 0, s_warp, &n_act);
  const int ng = (cnt + kGroup - 1) / kGroup;
  const int goff = block_exclusive_scan(ng, s_warp, &n_grp);
  if (threadIdx.x < Et) {
    rb.seg_offsets[threadIdx.x] = off;
    if (cnt > 0) rb.active[1 + aidx] = threadIdx.x;
    write_groups(rb, threadIdx.x, off, cnt, goff);
  }
  if (threadIdx.x == 0) {
    rb.seg_offsets[Et] = total;
    rb.active[0] = n_act;
    rb.group_off[Et] = n_grp;
  }
  __syncthreads();
  if (threadIdx.x < Et) s_cnt[threadIdx.x] = off;  // segment starts
  __syncthreads();
  for (int pl = threadIdx.x; pl < np; pl += blockDim.x) {
    const size_t p = (size_t)t0 * kp + pl;
    const int e = s_ids[pl];
    const int pos = s_cnt[e] + rank_of(pl);
    rb.seg_pairs[pos] = (int)p;
    rb.pair_pos[p] = pos;
  }
}

// Scan stage (one CTA): exclusive prefix over chunks per expert, offsets over
// experts, active list.  chunk_counts becomes the base of each (chunk, e).
__global__ void __launch_bounds__(1024) route_scan_kernel(int E, int nchunks, RouteBuffers rb) {
  pdl_wait();
  __shared__ int s_warp[32];
  const int e = threadIdx.x;
  int tot = 0;
  // (8 chunks per turn: their loads are issued together instead of one
  // dependent load-store round trip per chunk)
  constexpr int kB = 8;
  if (e < E) {
    for (int c0 = 0; c0 < nchunks; c0 += kB) {
      int v[kB];
#pragma unroll
      for (int i = 0; i < kB; i++)
        v[i] = c0 + i < nchunks ? rb.chunk_counts[(size_t)(c0 + i) * E + e] : 0;
#pragma unroll
      for (int i = 0; i < kB; i++)
        if (c0 + i < nchunks) {
          rb.chunk_counts[(size_t)(c0 + i) * E + e] = tot;
          tot += v[i];
        }
    }
  }
  int total = 0, n_act = 0, n_grp = 0;
  const int off = block_exclusive_scan(tot, s_warp, &total);
  const int aidx = block_exclusive_scan(tot > 0 ? 1 : 0, s_warp, &n_act);
  const int ng = (tot + kGroup - 1) / kGroup;
  const int goff = block_exclusive_scan(ng, s_warp, &n_grp);
  if (e < E) {
    rb.seg_offsets[e] = off;
    if (tot > 0) rb.active[1 + aidx] = e;
    for (int c0 = 0; c0 < nchunks; c0 += kB) {
      int v[kB];
#pragma unroll
      for (int i = 0; i < kB; i++)
        v[i] = c0 + i < nchunks ? rb.chunk_counts[(size_t)(c0 + i) * E + e] : 0;
#pragma unroll
      for (int i = 0; i < kB; i++)
        if (c0 + i < nchunks) rb.chunk_counts[(size_t)(c0 + i) * E + e] = v[i] + off;
    }
    write_groups(rb, e, off, tot, goff);
  }
  if (threadIdx.x == 0) {
    rb.seg_offsets[E] = total;
    rb.active[0] = n_act;
    rb.group_off[E] = n_grp;
  }
}

__global__ void __launch_bounds__(256) route_scatter_kernel(int T, int E, int k, RouteBuffers rb) {
  pdl_wait();
  const int chunk = blockIdx.x;
  const int t0 = chunk * kRouteChunk;
  const int nt = min(kRouteChunk, T - t0);
  for (int pl = threadIdx.x; pl < nt * k; pl += blockDim.x) {
    const size_t p = (size_t)t0 * k + pl;
    const int e = rb.ids[p];
    if (e < 0 || e >= E) {
      atomicOr(rb.status, kStatusBadExpert);
      continue;
    }
    const int pos = rb.chunk_counts[(size_t)chunk * E + e] + rb.rank[p];
    rb.seg_pairs[pos] = (int)p;
    rb.pair_pos[p] = pos;
  }
}

__global__ void route_empty_kernel(int E, RouteBuffers rb) {
  pdl_wait();
  if (threadIdx.x == 0) *rb.status = 0;  // (as route_chunk_kernel)
  for (int e = threadIdx.x; e <= E; e += blockDim.x) {
    rb.seg_offsets[e] = 0;
    rb.group_off[e] = 0;
  }
  if (threadIdx.x == 0) rb.active[0] = 0;
}

template <int MAXPL>
cudaError_t launch_chunks(const float* logits, int T, int E, int k, int sh, const RouteBuffers& rb,
                          int nchunks, cudaStream_t st) {
  // a warp per token for the top-k (in turns past 32 tokens); one chunk also
  // needs a thread per expert for its scans, and no more warps than either
  // (fewer warps make the CTA's barriers cheaper)
  int threads = 1024;
  if (nchunks == 1) {
    const int need_e = (E + sh + 31) / 32 * 32, need_t = 32 * (T < 32 ? T : 32);
    threads = need_e > need_t ? need_e : need_t;
  }
  const cudaError_t err = launch_pdl(route_chunk_kernel<MAXPL>, dim3(nchunks), dim3(threads), 0, st,
                                     logits, T, E, k, sh, rb, (int)(nchunks == 1));
  note_launches(1);
  return err;
}

}  // namespace

static size_t align256(size_t b) { return (b + 255) & ~(size_t)255; }

size_t route_scratch_bytes(int T, int E, int top_k) {
  const size_t P = (size_t)T * top_k;
  const size_t nchunks = (T + kRouteChunk - 1) / kRouteChunk;
  size_t b = 0;
  b += align256(sizeof(int32_t) * 4);            // status
  b += align256(sizeof(int32_t) * P);            // pair_pos
  b += align256(sizeof(int32_t) * (E + 1));      // active
  b += align256(sizeof(int32_t) * nchunks * E);  // chunk counts
  b += align256(sizeof(int32_t) * P);            // rank
  b += align256(sizeof(int32_t) * (E + 1));      // group_off
  b += align256(sizeof(int32_t) * 4 * max_groups(T, E, top_k));  // groups
  return b;
}

void route_carve(void* ws, int T, int E, int top_k, RouteBuffers* rb) {
  const size_t P = (size_t)T * top_k;
  const size_t nchunks = (T + kRouteChunk - 1) / kRouteChunk;
  char* p = static_cast<char*>(ws);
  rb->status = reinterpret_cast<int32_t*>(p);
  p += align256(sizeof(int32_t) * 4);
  rb->pair_pos = reinterpret_cast<int32_t*>(p);
  p += align256(sizeof(int32_t) * P);
  rb->active = reinterpret_cast<int32_t*>(p);
  p += align256(sizeof(int32_t) * (E + 1));
  rb->chunk_counts = reinterpret_cast<int32_t*>(p);
  p += align256(sizeof(int32_t) * nchunks * E);
  rb->rank = reinterpret_cast<int32_t*>(p);
  p += align256(sizeof(int32_t) * P);
  rb->group_off = reinterpret_cast<int32_t*>(p);
  p += align256(sizeof(int32_t) * (E + 1));
  rb->groups = reinterpret_cast<int32_t*>(p);
}

cudaError_t launch_route(const float* logits, int T, int E, int k, const RouteBuffers& rb,
                         cudaStream_t st, int shared) {
  const int sh = shared ? 1 : 0;
  if (T == 0) {
    const cudaError_t e = launch_pdl(route_empty_kernel, dim3(1), dim3(256), 0, st, E + sh, rb);
    note_launches(1);
    return e;
  }
  const int nchunks = (T + kRouteChunk - 1) / kRouteChunk;
  const int pl = (E + 31) / 32;
  cudaError_t err;
  if (pl <= 1) err = launch_chunks<1>(logits, T, E, k, sh, rb, nchunks, st);
  else if (pl <= 2) err = launch_chunks<2>(logits, T, E, k, sh, rb, nchunks, st);
  else if (pl <= 4) err = launch_chunks<4>(logits, T, E, k, sh, rb, nchunks, st);
  else if (pl <= 9) err = launch_chunks<9>(logits, T, E, k, sh, rb, nchunks, st);
  else if (pl <= 16) err = launch_chunks<16>(logits, T, E, k, sh, rb, nchunks, st);
  else err = launch_chunks<32>(logits, T, E, k, sh, rb, nchunks, st);
  if (err != cudaSuccess || nchunks == 1) return err;
  err = launch_pdl(route_scan_kernel, dim3(1), dim3(1024), 0, st, E + sh, nchunks, rb);
  note_launches(1);
  if (err != cudaSuccess) return err;
  err = launch_pdl(route_scatter_kernel, dim3(nchunks), dim3(256), 0, st, T, E + sh, k + sh, rb);
  note_launches(1);
  return err;
}

}  // namespace exl3
