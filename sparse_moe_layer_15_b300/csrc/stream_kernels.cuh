// Streaming (decode-size) path of the Flint MoE layer, T <= STREAM_MAX_T tokens.
//
// At decode sizes the layer is bound by reading weights: each touched expert's 6 MB and
// the shared expert's 12 MB are read once, the arithmetic is tiny.  So every weight tile is
// moved by one TMA copy into shared memory and consumed there by CUDA cores, and the work
// is split into enough independent tiles (column chunks x K splits) to keep all SMs
// streaming.  Split-K sums are reduced deterministically by the last tile of each chunk to
// arrive (an integer ticket, no floating-point atomics).
//
//   stream_k1: router (8-CTA clusters, one cluster per 4 tokens; scores reduced over the
//              cluster in distributed shared memory), top-6 + renormalisation, the
//              expert permutation (last cluster), L2 prefetch of the touched experts;
//              and, in other CTAs of the same grid, the shared expert's gate/up.
//   stream_k2: routed gate/up with fused SiLU-mul (touched experts only) and the shared
//              expert's down projection.
//   stream_k3: routed down projection scaled by the gate, and the combine
//              y = S + sum_j Y[inv(t, j)] in slot order (last tile of each column chunk).
#pragma once

#include <cooperative_groups.h>

#include "common.cuh"

namespace flint {
namespace cg = cooperative_groups;

constexpr int NTHREADS = 256;
constexpr int NWARPS = NTHREADS / 32;
constexpr int STREAM_MAX_T = 256;
constexpr int NT_MAX = 8;  // tokens per register block

constexpr int RT_TOK = 4;                // tokens per router cluster
constexpr int RT_CL = 8;                 // CTAs per router cluster (K split of H)
constexpr int RT_KR = H / RT_CL;         // 256 router rows per CTA
constexpr int SGU_KS = 8;                // shared gate/up: K splits
constexpr int SGU_KR = H / SGU_KS;       // 256
constexpr int SGU_NCH = IS / 64;         // 16 column chunks
constexpr int SGU_UNITS = SGU_KS * SGU_NCH;
constexpr int GU_KS = 8;                 // routed gate/up: K splits
constexpr int GU_KR = H / GU_KS;         // 256
constexpr int GU_NCH = I / 64;           // 8 column chunks
constexpr int GU_UPE = GU_KS * GU_NCH;   // 64 tiles per expert
constexpr int SD_KS = 4;                 // shared down: K splits
constexpr int SD_KR = IS / SD_KS;        // 256
constexpr int SD_NCH = H / 64;           // 32 column chunks
constexpr int SD_UNITS = SD_KS * SD_NCH; // 128
constexpr int DN_NCH = H / 64;           // routed down: 32 column chunks per expert, all I rows
constexpr int BOX_ROWS = 256;            // rows per TMA box of a weight tile (64 columns wide)

static_assert(SGU_UNITS % RT_CL == 0, "shared gate/up tiles must fill whole clusters");

struct StreamMaps {
  CUtensorMap wg;   // w_gate as [E*H][I]
  CUtensorMap wu;   // w_up   as [E*H][I]
  CUtensorMap wd;   // w_down as [E*I][H]
  CUtensorMap wsg;  // [H][IS]
  CUtensorMap wsu;  // [H][IS]
  CUtensorMap wsd;  // [IS][H]
};

// ---------------------------------------------------------------- shared-memory layouts
constexpr int TILE_BYTES = BOX_ROWS * 64 * 2;  // 32 KB per TMA box

struct SmemGU {  // gate/up tile (routed or shared): two KR x 64 tiles
  static constexpr int tiles = 0;                                   // 2 * 32 KB
  static constexpr int xs = tiles + 2 * TILE_BYTES;                 // [NT_MAX][256] f32
  static constexpr int red = xs + NT_MAX * 256 * 4;                 // [8][NT_MAX][128] f32
  static constexpr int out = red + NWARPS * NT_MAX * 128 * 4;       // [NT_MAX][128] f32
  static constexpr int bar = out + NT_MAX * 128 * 4;                // mbarrier
  static constexpr int flag = bar + 16;
  static constexpr int bytes = flag + 16;
};
struct SmemSD {  // shared down tile: one 256 x 64 tile
  static constexpr int tiles = 0;
  static constexpr int xs = tiles + TILE_BYTES;
  static constexpr int red = xs + NT_MAX * 256 * 4;
  static constexpr int out = red + NWARPS * NT_MAX * 64 * 4;
  static constexpr int bar = out + NT_MAX * 64 * 4;
  static constexpr int flag = bar + 16;
  static constexpr int bytes = flag + 16;
};
struct SmemDN {  // routed down tile: one 512 x 64 tile (two boxes)
  static constexpr int tiles = 0;
  static constexpr int xs = tiles + 2 * TILE_BYTES;                 // [NT_MAX][512] f32
  static constexpr int red = xs + NT_MAX * 512 * 4;
  static constexpr int out = red + NWARPS * NT_MAX * 64 * 4;
  static constexpr int bar = out + NT_MAX * 64 * 4;
  static constexpr int flag = bar + 16;
  static constexpr int bytes = flag + 16;
};
struct SmemRT {  // router CTA + the permutation
  static constexpr int xs = 0;                                      // [RT_TOK][256] f32
  static constexpr int red = xs + RT_TOK * RT_KR * 4;               // [8][RT_TOK][256] f32
  static constexpr int part = red + NWARPS * RT_TOK * E * 4;        // [RT_TOK][256] f32
  static constexpr int scores = part + RT_TOK * E * 4;              // [RT_TOK][256] f32
  static constexpr int flag = scores + RT_TOK * E * 4;
  static constexpr int bytes = flag + 16;
  // permutation scratch aliases `red` (used only after the router is done)
  static constexpr int s_cnt = red;                 // [E] int
  static constexpr int s_off = s_cnt + E * 4;       // [E+1] int (+pad)
  static constexpr int s_fill = s_off + (E + 4) * 4;// [E] int
  static constexpr int s_wcnt = s_fill + E * 4;     // [8][E] int
  static constexpr int s_wsum = s_wcnt + NWARPS * E * 4;  // [2][8] int
};
static_assert(SmemRT::s_wsum + 64 <= SmemRT::part, "permutation scratch must fit in the router buffer");

constexpr int cmax(int a, int b) { return a > b ? a : b; }
constexpr int K1_SMEM = cmax(SmemGU::bytes, SmemRT::bytes) + 1024;
constexpr int K2_SMEM = cmax(SmemGU::bytes, SmemSD::bytes) + 1024;
constexpr int K3_SMEM = SmemDN::bytes + 1024;

__device__ __forceinline__ uint8_t* aligned_smem(uint8_t* raw) {
  uint32_t a = smem_u32(raw);
  uint32_t pad = (1024u - (a & 1023u)) & 1023u;
  return raw + pad;
}

// ---------------------------------------------------------------- tile multiply-accumulate
// out[t][m*64 + c] = sum over the KR rows r of xs[t][r] * tile_m[r][c], for NT staged input
// rows and NM weight tiles (each KR x 64 bf16, row-major, in shared memory).  Each lane
// accumulates 8 columns of one row in four, rows ascending; the four row lanes are summed by
// a fixed shuffle tree, the eight warps in warp order: the result is bitwise reproducible.
template <int NT, int NM, int KR>
__device__ __forceinline__ void mac_block(const bf16* __restrict__ wt, const float* __restrict__ xs,
                                          float* __restrict__ red, float* __restrict__ out) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int rsub = lane >> 3, ch = lane & 7;
  constexpr int RPW = KR / NWARPS;  // rows per warp
  float acc[NT][NM][8];
#pragma unroll
  for (int t = 0; t < NT; ++t)
#pragma unroll
    for (int m = 0; m < NM; ++m)
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[t][m][q] = 0.f;

#pragma unroll 4
  for (int i = 0; i < RPW / 4; ++i) {
    const int r = warp * RPW + i * 4 + rsub;
    float xv[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) xv[t] = xs[t * KR + r];
#pragma unroll
    for (int m = 0; m < NM; ++m) {
      const uint4 w = *reinterpret_cast<const uint4*>(wt + (size_t)m * KR * 64 + r * 64 + ch * 8);
      float wf[8];
      bf16x8_to_f32(w, wf);
#pragma unroll
      for (int t = 0; t < NT; ++t)
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[t][m][q] = fmaf(xv[t], wf[q], acc[t][m][q]);
    }
  }
#pragma unroll
  for (int t = 0; t < NT; ++t)
#pragma unroll
    for (int m = 0; m < NM; ++m)
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        float v = acc[t][m][q];
        v += __shfl_xor_sync(0xffffffffu, v, 8);
        v += __shfl_xor_sync(0xffffffffu, v, 16);
        if (rsub == 0) red[((warp * NT + t) * NM + m) * 64 + ch * 8 + q] = v;
      }
  __syncthreads();
  for (int o = threadIdx.x; o < NT * NM * 64; o += NTHREADS) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < NWARPS; ++w) s += red[w * NT * NM * 64 + o];
    out[o] = s;
  }
  __syncthreads();
}

// Runs mac_block over `ntok` input rows in register blocks of up to NT_MAX tokens.
//   stage(xs, t0, nt, ntb): fill xs[t][r] (t < ntb, zero rows beyond nt), KR floats per row
//   store(out, t0, nt):     consume out[t][NM*64] for t < nt
template <int NM, int KR, class Stage, class Store>
__device__ __forceinline__ void mac_tokens(const bf16* wt, float* xs, float* red, float* out, int ntok,
                                           Stage stage, Store store) {
  for (int t0 = 0; t0 < ntok; t0 += NT_MAX) {
    const int nt = min(NT_MAX, ntok - t0);
    const int ntb = nt <= 1 ? 1 : nt <= 2 ? 2 : nt <= 4 ? 4 : 8;
    stage(xs, t0, nt, ntb);
    __syncthreads();
    switch (ntb) {
      case 1: mac_block<1, NM, KR>(wt, xs, red, out); break;
      case 2: mac_block<2, NM, KR>(wt, xs, red, out); break;
      case 4: mac_block<4, NM, KR>(wt, xs, red, out); break;
      default: mac_block<8, NM, KR>(wt, xs, red, out); break;
    }
    store(out, t0, nt);
    __syncthreads();
  }
}

// xs[t][r] = float(src_row(t)[k0 + r]) for r < KR, rows t < nt; zero for nt <= t < ntb.
template <int KR, class RowPtr>
__device__ __forceinline__ void stage_rows(float* xs, int nt, int ntb, int k0, RowPtr row_ptr) {
  constexpr int CPR = KR / 8;  // 16-byte chunks per row
  for (int c = threadIdx.x; c < ntb * CPR; c += NTHREADS) {
    const int t = c / CPR, q = c % CPR;
    float f[8];
    if (t < nt) {
      const uint4 v = *reinterpret_cast<const uint4*>(row_ptr(t) + k0 + q * 8);
      bf16x8_to_f32(v, f);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) f[j] = 0.f;
    }
    float4* d = reinterpret_cast<float4*>(xs + t * KR + q * 8);
    d[0] = make_float4(f[0], f[1], f[2], f[3]);
    d[1] = make_float4(f[4], f[5], f[6], f[7]);
  }
}

// Arrive on a ticket after this CTA's global writes; returns (in every thread) whether this
// CTA is the last of `total` arrivals, and if so resets the ticket for the next use.
__device__ __forceinline__ bool ticket_arrive(uint32_t* ticket, uint32_t total, int* s_flag) {
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint32_t old = atomicAdd(ticket, 1u);
    const bool last = (old == total - 1);
    if (last) atomicExch(ticket, 0u);
    *s_flag = last ? 1 : 0;
  }
  __syncthreads();
  const bool last = *s_flag != 0;
  if (last) __threadfence();
  return last;
}

// ================================================================ K1: router + shared gate/up
__device__ void router_cluster(const Params& p, uint8_t* sm, int cl, int rank);
__device__ void permute_small(const Params& p, uint8_t* sm);

__device__ void shared_gate_up_tile(const Params& p, const StreamMaps& maps, uint8_t* sm, int unit) {
  const int c = unit % SGU_NCH, s = unit / SGU_NCH;
  const int col0 = c * 64, k0 = s * SGU_KR;
  bf16* tiles = reinterpret_cast<bf16*>(sm + SmemGU::tiles);
  float* xs = reinterpret_cast<float*>(sm + SmemGU::xs);
  float* red = reinterpret_cast<float*>(sm + SmemGU::red);
  float* out = reinterpret_cast<float*>(sm + SmemGU::out);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + SmemGU::bar);
  int* flag = reinterpret_cast<int*>(sm + SmemGU::flag);
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(bar, 2 * TILE_BYTES);
    tma_load_2d(tiles, &maps.wsg, col0, k0, bar);
    tma_load_2d(tiles + BOX_ROWS * 64, &maps.wsu, col0, k0, bar);
  }
  pdl_wait();
  __syncthreads();
  if (!mbar_wait_bounded(bar, 0, p.status)) return;
  const int T = p.T;
  mac_tokens<2, SGU_KR>(
      tiles, xs, red, out, T,
      [&](float* xsb, int t0, int nt, int ntb) {
        stage_rows<SGU_KR>(xsb, nt, ntb, k0, [&](int t) { return p.xin + (size_t)(t0 + t) * H; });
      },
      [&](const float* o, int t0, int nt) {
        for (int q = threadIdx.x; q < nt * 128; q += NTHREADS) {
          const int t = q / 128, j = q % 128;
          p.P_sgu[((size_t)s * STREAM_MAX_T + t0 + t) * (2 * IS) + c * 128 + j] = o[q];
        }
      });
  if (!ticket_arrive(p.tickets + TicketLayout::sgu + c, SGU_KS, flag)) return;
  for (int q = threadIdx.x; q < T * 64; q += NTHREADS) {
    const int t = q / 64, j = q % 64;
    float g = 0.f, u = 0.f;
    for (int ss = 0; ss < SGU_KS; ++ss) {
      const float* P = p.P_sgu + ((size_t)ss * STREAM_MAX_T + t) * (2 * IS) + c * 128;
      g += __ldcg(P + j);
      u += __ldcg(P + 64 + j);
    }
    p.hs[(size_t)t * IS + col0 + j] = __float2bfloat16_rn(silu_f32(g) * u);
  }
}

__global__ void __cluster_dims__(RT_CL, 1, 1) __launch_bounds__(NTHREADS)
    stream_k1(const __grid_constant__ Params p, const __grid_constant__ StreamMaps maps, int n_router_ctas, int with_shared) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = aligned_smem(smem_raw);
  pdl_launch_dependents();
  if ((int)blockIdx.x < n_router_ctas) {
    pdl_wait();
    router_cluster(p, sm, blockIdx.x / RT_CL, blockIdx.x % RT_CL);
  } else if (with_shared) {
    shared_gate_up_tile(p, maps, sm, blockIdx.x - n_router_ctas);
  }
}

__device__ void router_cluster(const Params& p, uint8_t* sm, int cl, int rank) {
  cg::cluster_group cluster = cg::this_cluster();
  float* xs = reinterpret_cast<float*>(sm + SmemRT::xs);
  float* red = reinterpret_cast<float*>(sm + SmemRT::red);
  float* part = reinterpret_cast<float*>(sm + SmemRT::part);
  float* scores = reinterpret_cast<float*>(sm + SmemRT::scores);
  int* flag = reinterpret_cast<int*>(sm + SmemRT::flag);
  const int t0 = cl * RT_TOK;
  const int nt = min(RT_TOK, p.T - t0);
  const int k0 = rank * RT_KR;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  // stage the token rows of this K slice
  stage_rows<RT_KR>(xs, nt, RT_TOK, k0, [&](int t) { return p.xin + (size_t)(t0 + t) * H; });
  __syncthreads();

  // partial logits: lane owns experts 8*lane..8*lane+7, warp owns rows warp, warp+8, ...
  float acc[RT_TOK][8];
#pragma unroll
  for (int t = 0; t < RT_TOK; ++t)
#pragma unroll
    for (int q = 0; q < 8; ++q) acc[t][q] = 0.f;
  const bf16* wr = p.w_router + (size_t)k0 * E + lane * 8;
#pragma unroll 8
  for (int i = 0; i < RT_KR / NWARPS; ++i) {
    const int r = warp + i * NWARPS;
    const uint4 w = __ldg(reinterpret_cast<const uint4*>(wr + (size_t)r * E));
    float wf[8];
    bf16x8_to_f32(w, wf);
#pragma unroll
    for (int t = 0; t < RT_TOK; ++t) {
      const float xv = xs[t * RT_KR + r];
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[t][q] = fmaf(xv, wf[q], acc[t][q]);
    }
  }
#pragma unroll
  for (int t = 0; t < RT_TOK; ++t)
#pragma unroll
    for (int q = 0; q < 8; ++q) red[(warp * RT_TOK + t) * E + lane * 8 + q] = acc[t][q];
  __syncthreads();
  {
    const int e = threadIdx.x;  // NTHREADS == E
#pragma unroll
    for (int t = 0; t < RT_TOK; ++t) {
      float s = 0.f;
#pragma unroll
      for (int w = 0; w < NWARPS; ++w) s += red[(w * RT_TOK + t) * E + e];
      part[t * E + e] = s;
    }
  }
  cluster.sync();
  // CTA `rank` finishes experts [32*rank, 32*rank + 32): sum the 8 K slices in rank order,
  // add the bias, apply the sigmoid and deposit the score in CTA 0.
  {
    float* scores0 = cluster.map_shared_rank(scores, 0);
    for (int q = threadIdx.x; q < nt * 32; q += NTHREADS) {
      const int t = q / 32, e = rank * 32 + (q % 32);
      float l = 0.f;
#pragma unroll
      for (int r = 0; r < RT_CL; ++r) l += cluster.map_shared_rank(part, r)[t * E + e];
      if (p.router_bias) l += p.router_bias[e];
      scores0[t * E + e] = 1.0f / (1.0f + expf(-l));
    }
  }
  cluster.sync();
  if (rank != 0) return;

  // top-K per token (warp t): key = (score bits, 255 - expert) -> max = highest score,
  // lowest index on equal scores.
  if (warp < nt) {
    const int t = warp;
    uint64_t key[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int e = lane + 32 * q;
      key[q] = (uint64_t(__float_as_uint(scores[t * E + e])) << 32) | uint32_t(E - 1 - e);
    }
    float sel_s[K];
    int sel_e[K];
#pragma unroll
    for (int j = 0; j < K; ++j) {
      uint64_t best = 0;
#pragma unroll
      for (int q = 0; q < 8; ++q) best = key[q] > best ? key[q] : best;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const uint64_t o = __shfl_xor_sync(0xffffffffu, best, off);
        best = o > best ? o : best;
      }
      const int e = E - 1 - int(best & 0xFFFFFFFFu);
      sel_e[j] = e;
      sel_s[j] = __uint_as_float(uint32_t(best >> 32));
      if ((e & 31) == lane) key[e >> 5] = 0;  // scores are >= 0, so 0 never wins again
    }
    if (lane == 0) {
      float sum = 0.f;
#pragma unroll
      for (int j = 0; j < K; ++j) sum += sel_s[j];
      const int tg = t0 + t;
#pragma unroll
      for (int j = 0; j < K; ++j) {
        const float g = sel_s[j] / sum;
        p.topk_idx[tg * K + j] = sel_e[j];
        p.topk_w[tg * K + j] = g;
        if (p.out_idx) p.out_idx[tg * K + j] = sel_e[j];
        if (p.out_w) p.out_w[tg * K + j] = g;
      }
    }
  }
  const int n_clusters = (p.T + RT_TOK - 1) / RT_TOK;
  if (!ticket_arrive(p.tickets + TicketLayout::router, n_clusters, flag)) return;
  permute_small(p, sm);
}

// Stable counting sort of the T*K (token, slot) pairs by expert, in one CTA.
__device__ void permute_small(const Params& p, uint8_t* sm) {
  int* s_cnt = reinterpret_cast<int*>(sm + SmemRT::s_cnt);
  int* s_off = reinterpret_cast<int*>(sm + SmemRT::s_off);
  int* s_fill = reinterpret_cast<int*>(sm + SmemRT::s_fill);
  int* s_wcnt = reinterpret_cast<int*>(sm + SmemRT::s_wcnt);
  int* s_wsum = reinterpret_cast<int*>(sm + SmemRT::s_wsum);
  const int n = p.T * K;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  s_cnt[tid] = 0;
  __syncthreads();
  for (int q = tid; q < n; q += NTHREADS) {
    const int e = __ldcg(p.topk_idx + q);
    if (e < 0 || e >= E) {
      record_status(p.status, ST_BOUNDS);
      continue;
    }
    atomicAdd(&s_cnt[e], 1);
  }
  __syncthreads();
  // exclusive scans over experts (tid == expert) of the counts and of "touched" flags
  const int c = s_cnt[tid];
  const int f = c > 0 ? 1 : 0;
  int ic = c, jf = f;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int a = __shfl_up_sync(0xffffffffu, ic, off);
    const int b = __shfl_up_sync(0xffffffffu, jf, off);
    if (lane >= off) {
      ic += a;
      jf += b;
    }
  }
  if (lane == 31) {
    s_wsum[warp] = ic;
    s_wsum[NWARPS + warp] = jf;
  }
  __syncthreads();
  int bc = 0, bf = 0;
  for (int w = 0; w < warp; ++w) {
    bc += s_wsum[w];
    bf += s_wsum[NWARPS + w];
  }
  const int off_e = bc + ic - c;
  const int pos = bf + jf - f;
  s_off[tid] = off_e;
  s_fill[tid] = off_e;
  p.counts[tid] = c;
  p.offsets[tid] = off_e;
  if (p.out_counts) p.out_counts[tid] = c;
  if (f) p.touched[pos] = tid;
  if (tid == NTHREADS - 1) {
    p.offsets[E] = off_e + c;
    *p.n_touched = pos + f;
    s_wsum[2 * NWARPS] = pos + f;
  }
  __syncthreads();
  // stable scatter, 256 pairs at a time in (t, j) order
  for (int base = 0; base < n; base += NTHREADS) {
    for (int q = tid; q < NWARPS * E; q += NTHREADS) s_wcnt[q] = 0;
    __syncthreads();
    const int pi = base + tid;
    int e = pi < n ? __ldcg(p.topk_idx + pi) : -1;
    if (e >= E) e = -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int r = __popc(peers & ((1u << lane) - 1u));
    if (e >= 0 && r == 0) s_wcnt[warp * E + e] = __popc(peers);
    __syncthreads();
    if (e >= 0) {
      int before = 0;
      for (int w = 0; w < warp; ++w) before += s_wcnt[w * E + e];
      const int row = s_fill[e] + before + r;
      p.perm[row] = pi;
      p.inv[pi] = row;
    }
    __syncthreads();
    {
      int add = 0;
      for (int w = 0; w < NWARPS; ++w) add += s_wcnt[w * E + tid];
      s_fill[tid] += add;
    }
    __syncthreads();
  }
  // L2 prefetch of the touched experts' weights when they fit the budget
  const int nt_exp = s_wsum[2 * NWARPS];
  const unsigned long long per_expert = 3ull * H * I * 2;
  if ((unsigned long long)nt_exp * per_expert <= p.prefetch_bytes_max) {
    constexpr uint32_t CH = 64 * 1024;
    constexpr int CHUNKS = (H * I * 2) / CH;  // 32 chunks of each 2 MB matrix
    for (int q = tid; q < nt_exp * 3 * CHUNKS; q += NTHREADS) {
      const int u = q / (3 * CHUNKS), m = (q / CHUNKS) % 3, cc = q % CHUNKS;
      const int e = p.touched[u];
      const bf16* base = m == 0 ? p.w_gate : m == 1 ? p.w_up : p.w_down;
      prefetch_l2_bulk(reinterpret_cast<const uint8_t*>(base + (size_t)e * H * I) + (size_t)cc * CH, CH);
    }
  }
}

// ================================================================ K2: routed gate/up + shared down
__device__ void routed_gate_up_tile(const Params& p, const StreamMaps& maps, uint8_t* sm, int unit) {
  const int u = unit / GU_UPE;
  const int c = unit % GU_NCH, s = (unit / GU_NCH) % GU_KS;
  bf16* tiles = reinterpret_cast<bf16*>(sm + SmemGU::tiles);
  float* xs = reinterpret_cast<float*>(sm + SmemGU::xs);
  float* red = reinterpret_cast<float*>(sm + SmemGU::red);
  float* out = reinterpret_cast<float*>(sm + SmemGU::out);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + SmemGU::bar);
  int* flag = reinterpret_cast<int*>(sm + SmemGU::flag);
  pdl_wait();
  if (u >= __ldcg(p.n_touched)) return;
  const int e = __ldcg(p.touched + u);
  const int off = __ldcg(p.offsets + e), n = __ldcg(p.counts + e);
  const int col0 = c * 64, k0 = s * GU_KR;
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(bar, 2 * TILE_BYTES);
    tma_load_2d(tiles, &maps.wg, col0, e * H + k0, bar);
    tma_load_2d(tiles + BOX_ROWS * 64, &maps.wu, col0, e * H + k0, bar);
  }
  __syncthreads();
  if (!mbar_wait_bounded(bar, 0, p.status)) return;
  const int rows_cap = p.T * K;
  mac_tokens<2, GU_KR>(
      tiles, xs, red, out, n,
      [&](float* xsb, int t0, int nt, int ntb) {
        stage_rows<GU_KR>(xsb, nt, ntb, k0, [&](int t) {
          const int tok = __ldcg(p.perm + off + t0 + t) / K;
          return p.xin + (size_t)tok * H;
        });
      },
      [&](const float* o, int t0, int nt) {
        for (int q = threadIdx.x; q < nt * 128; q += NTHREADS) {
          const int t = q / 128, j = q % 128;
          p.P_gu[((size_t)s * rows_cap + off + t0 + t) * (2 * I) + c * 128 + j] = o[q];
        }
      });
  if (!ticket_arrive(p.tickets + TicketLayout::gu + e * GU_NCH + c, GU_KS, flag)) return;
  for (int q = threadIdx.x; q < n * 64; q += NTHREADS) {
    const int t = q / 64, j = q % 64;
    float g = 0.f, uu = 0.f;
    for (int ss = 0; ss < GU_KS; ++ss) {
      const float* P = p.P_gu + ((size_t)ss * rows_cap + off + t) * (2 * I) + c * 128;
      g += __ldcg(P + j);
      uu += __ldcg(P + 64 + j);
    }
    p.h[(size_t)(off + t) * I + col0 + j] = __float2bfloat16_rn(silu_f32(g) * uu);
  }
}

__device__ void shared_down_tile(const Params& p, const StreamMaps& maps, uint8_t* sm, int unit) {
  const int c = unit % SD_NCH, s = unit / SD_NCH;
  const int col0 = c * 64, k0 = s * SD_KR;
  bf16* tiles = reinterpret_cast<bf16*>(sm + SmemSD::tiles);
  float* xs = reinterpret_cast<float*>(sm + SmemSD::xs);
  float* red = reinterpret_cast<float*>(sm + SmemSD::red);
  float* out = reinterpret_cast<float*>(sm + SmemSD::out);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + SmemSD::bar);
  int* flag = reinterpret_cast<int*>(sm + SmemSD::flag);
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(bar, TILE_BYTES);
    tma_load_2d(tiles, &maps.wsd, col0, k0, bar);
  }
  pdl_wait();
  __syncthreads();
  if (!mbar_wait_bounded(bar, 0, p.status)) return;
  const int T = p.T;
  mac_tokens<1, SD_KR>(
      tiles, xs, red, out, T,
      [&](float* xsb, int t0, int nt, int ntb) {
        stage_rows<SD_KR>(xsb, nt, ntb, k0, [&](int t) { return p.hs + (size_t)(t0 + t) * IS; });
      },
      [&](const float* o, int t0, int nt) {
        for (int q = threadIdx.x; q < nt * 64; q += NTHREADS) {
          const int t = q / 64, j = q % 64;
          p.P_sd[((size_t)s * STREAM_MAX_T + t0 + t) * H + col0 + j] = o[q];
        }
      });
  if (!ticket_arrive(p.tickets + TicketLayout::sd + c, SD_KS, flag)) return;
  for (int q = threadIdx.x; q < T * 64; q += NTHREADS) {
    const int t = q / 64, j = q % 64;
    float v = 0.f;
    for (int ss = 0; ss < SD_KS; ++ss) v += __ldcg(p.P_sd + ((size_t)ss * STREAM_MAX_T + t) * H + col0 + j);
    p.S[(size_t)t * H + col0 + j] = v;
  }
}

__global__ void __launch_bounds__(NTHREADS)
    stream_k2(const __grid_constant__ Params p, const __grid_constant__ StreamMaps maps, int n_routed_ctas) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = aligned_smem(smem_raw);
  pdl_launch_dependents();
  if ((int)blockIdx.x < n_routed_ctas)
    routed_gate_up_tile(p, maps, sm, blockIdx.x);
  else
    shared_down_tile(p, maps, sm, blockIdx.x - n_routed_ctas);
}

// ================================================================ K3: routed down + combine
__global__ void __launch_bounds__(NTHREADS) stream_k3(const __grid_constant__ Params p, const __grid_constant__ StreamMaps maps) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = aligned_smem(smem_raw);
  pdl_launch_dependents();
  const int u = blockIdx.x / DN_NCH, c = blockIdx.x % DN_NCH;
  bf16* tiles = reinterpret_cast<bf16*>(sm + SmemDN::tiles);
  float* xs = reinterpret_cast<float*>(sm + SmemDN::xs);
  float* red = reinterpret_cast<float*>(sm + SmemDN::red);
  float* out = reinterpret_cast<float*>(sm + SmemDN::out);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + SmemDN::bar);
  int* flag = reinterpret_cast<int*>(sm + SmemDN::flag);
  pdl_wait();
  const int n_touched = __ldcg(p.n_touched);
  if (u >= n_touched) return;
  const int e = __ldcg(p.touched + u);
  const int off = __ldcg(p.offsets + e), n = __ldcg(p.counts + e);
  const int col0 = c * 64;
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(bar, 2 * TILE_BYTES);
    tma_load_2d(tiles, &maps.wd, col0, e * I, bar);
    tma_load_2d(tiles + BOX_ROWS * 64, &maps.wd, col0, e * I + BOX_ROWS, bar);
  }
  __syncthreads();
  if (!mbar_wait_bounded(bar, 0, p.status)) return;
  mac_tokens<1, I>(
      tiles, xs, red, out, n,
      [&](float* xsb, int t0, int nt, int ntb) {
        stage_rows<I>(xsb, nt, ntb, 0, [&](int t) { return p.h + (size_t)(off + t0 + t) * I; });
      },
      [&](const float* o, int t0, int nt) {
        for (int q = threadIdx.x; q < nt * 64; q += NTHREADS) {
          const int t = q / 64, j = q % 64;
          const int row = off + t0 + t;
          const float g = __ldcg(p.topk_w + __ldcg(p.perm + row));
          p.Y[(size_t)row * H + col0 + j] = g * o[q];
        }
      });
  if (!ticket_arrive(p.tickets + TicketLayout::dn + c, (uint32_t)n_touched, flag)) return;
  // combine of column chunk c: y = S + sum_j Y[inv(t, j)] (slot order) [+ x]
  const bool residual = (p.flags & 2u) != 0;
  for (int q = threadIdx.x; q < p.T * 64; q += NTHREADS) {
    const int t = q / 64, j = q % 64;
    float v = __ldcg(p.S + (size_t)t * H + col0 + j);
#pragma unroll
    for (int k = 0; k < K; ++k) v += __ldcg(p.Y + (size_t)__ldcg(p.inv + t * K + k) * H + col0 + j);
    if (residual) v += __bfloat162float(p.x[(size_t)t * H + col0 + j]);
    p.y[(size_t)t * H + col0 + j] = __float2bfloat16_rn(v);
  }
}

// ================================================================ K0: RMSNorm (pre-norm layers)
// xn[t] = bf16(x[t] / sqrt(mean(x[t]^2) + eps)), unit weight; one CTA per token.
__global__ void __launch_bounds__(NTHREADS) rmsnorm_kernel(const __grid_constant__ Params p) {
  __shared__ float s_w[NWARPS];
  pdl_launch_dependents();
  pdl_wait();
  const int t = blockIdx.x;
  const bf16* xr = p.x + (size_t)t * H;
  float f[8];
  const uint4 v = *reinterpret_cast<const uint4*>(xr + threadIdx.x * 8);
  bf16x8_to_f32(v, f);
  float ss = 0.f;
#pragma unroll
  for (int q = 0; q < 8; ++q) ss = fmaf(f[q], f[q], ss);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  if ((threadIdx.x & 31) == 0) s_w[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < NWARPS; ++w) tot += s_w[w];
  const float d = sqrtf(tot / float(H) + p.rms_eps);
  uint32_t packed[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const __nv_bfloat162 b = __floats2bfloat162_rn(f[2 * q] / d, f[2 * q + 1] / d);
    packed[q] = *reinterpret_cast<const uint32_t*>(&b);
  }
  *reinterpret_cast<uint4*>(p.xn + (size_t)t * H + threadIdx.x * 8) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
}

}  // namespace flint
