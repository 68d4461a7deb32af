// Prefill-size path of the Flint MoE layer (T > 256 tokens): the contractions are dense enough
// for the tensor cores, so every GEMM-shaped step runs on the tcgen05 engine (tc_gemm.cuh):
//
//   router    [T x 2048] x W_r [2048 x 256] (ROWS): epilogue = bias, top-6 by logit with the
//             lower index first on ties, sigmoid of the six, renormalised gates, and a
//             per-tile histogram of the choices;
//   scatter   SPLIT CTAs per 128-token tile: counts, offsets and the 256-row group prefix of
//             every expert (each CTA reduces the histograms itself), the stable (t, j)-order
//             placement of the pairs into expert-sorted rows (perm / inv), and the copied input
//             rows xs[row] = x[t];
//   gate/up   grouped over (expert, 64-column pair of gate and up, 256-row group) in COLUMNS
//             orientation (N = the group's rows rounded up to 16), then the shared expert over
//             (64-column pair, 256-token group): h = bf16(silu(g) * u);
//   down      grouped over (expert, 128 output columns, 256-row group), COLUMNS: epilogue
//             Yb[row] = bf16(gate(row) * acc); then the shared expert's down projection over
//             (128 output columns, 256-token group): S[t] = acc (fp32);
//   combine   y[t] = bf16(S[t] + sum_j Yb[inv(t, j)] in slot order (+ x[t])).
// An expert's tiles are numbered with the column block fastest: the CTAs working at the same time
// read whole weight rows (all column blocks of one row group) and the next row group of the
// expert finds its weights in L2.
#pragma once

#include "common.cuh"
#include "tc_gemm.cuh"

namespace flint {
namespace pf {

using tc::TileInfo;
using tc::TM;
using tc::tmem_ld32;
using tc::epi_sync;

constexpr int RG = 2 * TM;        // rows per COLUMNS tile (the MMA's N <= 256)
constexpr int NCT_GU = I / 64;    // 8 column pairs (64 of gate | 64 of up) of a routed gate/up
// (the shared gate/up has p.sw / 64 column pairs: 16 for the MoE's shared expert, 96 for a dense layer)
constexpr int NCT_DN = H / 128;   // 16 output column blocks of a down projection

struct Maps {
  CUtensorMap xin;  // [T][H], box 64 x 128 (router, ROWS tiles)
  CUtensorMap xin_c;  // [T][H], box 64 x 64 (shared gate/up, COLUMNS tiles)
  CUtensorMap xs;   // [6 max_T][H], box 64 x 64 (routed gate/up, COLUMNS tiles)
  CUtensorMap h;    // [6 max_T][I], box 64 x 64 (COLUMNS tiles)
  CUtensorMap hs;   // [max_T][sw], box 64 x 64 (COLUMNS tiles)
  CUtensorMap wr;   // [H][E], box 64 x 64 (B operand)
  CUtensorMap wg;   // [E H][I], box 64 x 64
  CUtensorMap wu;
  CUtensorMap wd;   // [E I][H], box 64 x 64
  CUtensorMap wsg;  // [H][sw], box 64 x 64
  CUtensorMap wsu;
  CUtensorMap wsd;  // [sw][H], box 64 x 64
};

__device__ __forceinline__ void store_bf16x32(bf16* dst, const float* v) {
  uint32_t w[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const __nv_bfloat162 b = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    w[i] = *reinterpret_cast<const uint32_t*>(&b);
  }
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int q = 0; q < 4; ++q) d[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
}

// ================================================================ router
struct RouterTC {
  static constexpr bool kColumns = false;
  Params p;
  CUtensorMap xin, wr;
  __device__ void prologue(uint8_t*) const {
    if ((p.flags & FLAG_TEST_WAIT_TIMEOUT) && blockIdx.x == 0 && threadIdx.x == 0) test_wait_timeout(p.status);
  }
  __device__ int num_tiles(const uint8_t*) const { return (p.T + TM - 1) / TM; }
  __device__ int kblocks() const { return H / tc::TK; }
  __device__ uint32_t* status() const { return p.status; }
  __device__ unsigned long long* trace() const { return p.trace ? p.trace + 16 : nullptr; }  // slots 16..23
  __device__ void tile(int i, TileInfo& t, const uint8_t*) const {
    t.amap = &xin;
    t.a_row0 = i * TM;
    t.b_row0 = 0;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      t.bmap[c] = &wr;
      t.bcol[c] = c * 64;
    }
    t.row0 = i * TM;
    t.valid = min(TM, p.T - i * TM);
    t.col0 = 0;
    t.aux = i;
  }
  // Thread `row` owns token row0 + row: its 256 logits (+ bias) stream out of TMEM 32 at a
  // time in expert order; a running top-6 keeps the higher logit, and on equal logits the
  // expert seen first (the lower index).  The sigmoid is strictly increasing, so this is the
  // order of the scores; ranking the fp32 logits also avoids the fp32 score saturating near 1.
  // Only the six chosen logits go through the sigmoid.
  __device__ void epilogue(const TileInfo& t, uint32_t trow, int row, uint8_t* epi, const uint8_t*) const {
    int* hist = reinterpret_cast<int*>(epi);
    hist[row] = 0;
    hist[row + TM] = 0;
    float l6[K];
    int e6[K];
#pragma unroll
    for (int j = 0; j < K; ++j) {
      l6[j] = -INFINITY;
      e6[j] = -1;
    }
#pragma unroll 1
    for (int c = 0; c < E / 32; ++c) {
      float v[32];
      tmem_ld32(trow + uint32_t(c * 32), v);
#pragma unroll
      for (int q = 0; q < 32; ++q) {
        const int e = c * 32 + q;
        float l = v[q];
        if (p.router_bias) l += p.router_bias[e];
        if (l > l6[K - 1]) {
          l6[K - 1] = l;
          e6[K - 1] = e;
#pragma unroll
          for (int j = K - 1; j > 0; --j) {
            if (l6[j] > l6[j - 1]) {
              const float tl = l6[j];
              l6[j] = l6[j - 1];
              l6[j - 1] = tl;
              const int te = e6[j];
              e6[j] = e6[j - 1];
              e6[j - 1] = te;
            }
          }
        }
      }
    }
    float s6[K];
#pragma unroll
    for (int j = 0; j < K; ++j) s6[j] = 1.0f / (1.0f + expf(-l6[j]));
    epi_sync();  // histogram zeroed
    if (row < t.valid) {
      float sum = 0.f;
#pragma unroll
      for (int j = 0; j < K; ++j) sum += s6[j];
      const int tok = t.row0 + row;
#pragma unroll
      for (int j = 0; j < K; ++j) {
        const float g = s6[j] / sum;
        p.topk_idx[tok * K + j] = e6[j];
        p.topk_w[tok * K + j] = g;
        if (p.out_idx) p.out_idx[tok * K + j] = e6[j];
        if (p.out_w) p.out_w[tok * K + j] = g;
        atomicAdd(&hist[e6[j]], 1);
      }
    }
    epi_sync();
    p.hist[(size_t)t.aux * E + row] = hist[row];
    p.hist[(size_t)t.aux * E + row + TM] = hist[row + TM];
    epi_sync();  // before the next tile clears the histogram
  }
};

// ================================================================ scan + scatter + gather
// SPLIT CTAs (256 threads) per 128-token tile.  Every CTA first reduces the router's per-tile
// histograms itself -- thread e sums hist[.][e] over all tiles (count of expert e) and over the
// tiles before its own (rows of e that earlier tiles take) -- and scans the counts over the
// experts (offsets, and the RG-row group prefix mtp used by the grouped GEMMs); CTA 0 writes
// those tables.  Then the tile's 768 (t, j) pairs in order get their expert-sorted rows
// (stable: token order, then slot order, within an expert), and each CTA copies its share of
// the input rows, xs[row] = x[t] (TMA then reads them as 64-row boxes; a row gather in the
// GEMM's producer with cp.async could not keep enough bytes in flight).  `place` = 0 runs the
// tables only (one CTA: routing alone).
constexpr int SPLIT = 4;

__global__ void __launch_bounds__(256) scatter_kernel(const __grid_constant__ Params p, int place) {
  __shared__ int s_fill[E];
  __shared__ int s_wcnt[8][E];
  __shared__ int s_rows[TM * K];
  __shared__ int s_w[2][8];
  pdl_launch_dependents();
  pdl_wait();
  const int tile = blockIdx.x / SPLIT, part = blockIdx.x % SPLIT;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int ntiles = (p.T + TM - 1) / TM;
  // ---- counts and this tile's base rows: independent loads, 16 in flight per thread
  int tot = 0, pre = 0;
  for (int t0 = 0; t0 < ntiles; t0 += 16) {
    int v[16];
#pragma unroll
    for (int q = 0; q < 16; ++q) v[q] = t0 + q < ntiles ? __ldcg(p.hist + (size_t)(t0 + q) * E + tid) : 0;
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      tot += v[q];
      if (t0 + q < tile) pre += v[q];
    }
  }
  // ---- exclusive scans over the experts of the counts and of their RG-row group counts
  const int mt = (tot + RG - 1) / RG;
  int ic = tot, im = mt;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int a = __shfl_up_sync(0xffffffffu, ic, off);
    const int b = __shfl_up_sync(0xffffffffu, im, off);
    if (lane >= off) {
      ic += a;
      im += b;
    }
  }
  if (lane == 31) {
    s_w[0][warp] = ic;
    s_w[1][warp] = im;
  }
  __syncthreads();
  int bc = 0, bm = 0;
  for (int w = 0; w < warp; ++w) {
    bc += s_w[0][w];
    bm += s_w[1][w];
  }
  const int off_e = bc + ic - tot;
  if (blockIdx.x == 0) {
    p.counts[tid] = tot;
    p.offsets[tid] = off_e;
    p.mtp[tid] = bm + im - mt;
    if (p.out_counts) p.out_counts[tid] = tot;
    if (tid == E - 1) {
      p.offsets[E] = off_e + tot;
      p.mtp[E] = bm + im;
    }
  }
  if (!place) return;
  s_fill[tid] = off_e + pre;
  __syncthreads();
  // ---- stable placement of the tile's pairs
  const int t0 = tile * TM;
  const int npairs = min(TM, p.T - t0) * K;
  for (int base = 0; base < npairs; base += 256) {
    for (int q = tid; q < 8 * E; q += 256) (&s_wcnt[0][0])[q] = 0;
    __syncthreads();
    const int pi = base + tid;
    int e = pi < npairs ? __ldcg(p.topk_idx + t0 * K + pi) : -1;
    if (e >= E) {
      record_status(p.status, ST_BOUNDS);
      e = -1;
    }
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int r = __popc(peers & ((1u << lane) - 1u));
    if (e >= 0 && r == 0) s_wcnt[warp][e] = __popc(peers);
    __syncthreads();
    if (e >= 0) {
      int before = 0;
      for (int w = 0; w < warp; ++w) before += s_wcnt[w][e];
      const int row = s_fill[e] + before + r;
      if (part == 0) {
        p.perm[row] = t0 * K + pi;
        p.inv[t0 * K + pi] = row;
      }
      s_rows[pi] = row;
    } else if (pi < npairs) {
      s_rows[pi] = -1;
    }
    __syncthreads();
    int add = 0;
    for (int w = 0; w < 8; ++w) add += s_wcnt[w][tid];
    s_fill[tid] += add;
    __syncthreads();
  }
  // ---- gather: this CTA's contiguous share of the pairs; a warp copies two 4 KB rows at a
  // time (16 loads of 16 bytes in flight per lane)
  const int per = (npairs + SPLIT - 1) / SPLIT;
  const int qb = part * per, qe = min(npairs, qb + per);
  constexpr int V = H / 8 / 32;  // uint4 per lane per row
  for (int q = qb + warp; q < qe; q += 16) {
    const int q2 = q + 8;
    const bool two = q2 < qe;
    uint4 a[V], b[V];
    const uint4* sa = reinterpret_cast<const uint4*>(p.xin + (size_t)(t0 + q / K) * H);
    const uint4* sb = reinterpret_cast<const uint4*>(p.xin + (size_t)(t0 + (two ? q2 : q) / K) * H);
#pragma unroll
    for (int k = 0; k < V; ++k) a[k] = __ldg(sa + lane + 32 * k);
#pragma unroll
    for (int k = 0; k < V; ++k) b[k] = __ldg(sb + lane + 32 * k);
    const int ra = s_rows[q];
    if (ra >= 0) {
      uint4* d = reinterpret_cast<uint4*>(p.xs + (size_t)ra * H);
#pragma unroll
      for (int k = 0; k < V; ++k) d[lane + 32 * k] = a[k];
    }
    if (two) {
      const int rb = s_rows[q2];
      if (rb >= 0) {
        uint4* d = reinterpret_cast<uint4*>(p.xs + (size_t)rb * H);
#pragma unroll
        for (int k = 0; k < V; ++k) d[lane + 32 * k] = b[k];
      }
    }
  }
}

// Routing tables of the grouped GEMMs, copied to shared memory by every CTA: mtp[0..E] (prefix
// over the experts of their RG-row group counts), offsets[0..E].  A dense layer has no routed
// rows: all zero.
struct GroupTable {
  __device__ static void load(const Params& p, uint8_t* tbl) {
    int* mtp = reinterpret_cast<int*>(tbl);
    int* off = mtp + (E + 1);
    for (int i = threadIdx.x; i <= E; i += blockDim.x) {
      mtp[i] = p.dense ? 0 : __ldcg(p.mtp + i);
      off[i] = p.dense ? 0 : __ldcg(p.offsets + i);
    }
  }
  // expert whose tile range [per * mtp[e], per * mtp[e+1]) holds tile i
  __device__ static int find(const int* mtp, int per, int i) {
    int lo = 0, hi = E - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (mtp[mid] * per <= i)
        lo = mid;
      else
        hi = mid - 1;
    }
    return lo;
  }
};

// Position p of a list of R routed tiles followed by S shared-expert tiles: returns true and
// the shared tile's index, or false and the routed tile's index.  (Spreading the shared tiles
// evenly through the routed ones was measured slower: 0.746 vs 0.684 ms per layer at T = 8192.)
__device__ __forceinline__ bool shared_tile(int p, int R, int& idx) {
  if (p >= R) {
    idx = p - R;
    return true;
  }
  idx = p;
  return false;
}

// ================================================================ gate/up (routed + shared)
// COLUMNS tiles: 64 columns of gate (TMEM lanes 0..63) and the same 64 columns of up (lanes
// 64..127), and up to RG = 256 rows as the MMA's N (rounded up to 16): a routed expert's rows
// (expert-sorted copies, xs), so a ragged expert costs its own row count instead of whole
// 128-row tiles; then the shared expert over 256-token groups of the layer input.
struct GateUpTC {
  static constexpr bool kColumns = true;
  Params p;
  CUtensorMap xs, xin_c, wg, wu, wsg, wsu;
  __device__ void prologue(uint8_t* tbl) const { GroupTable::load(p, tbl); }
  __device__ int num_tiles(const uint8_t* tbl) const {
    const int* mtp = reinterpret_cast<const int*>(tbl);
    return NCT_GU * mtp[E] + (p.sw / 64) * ((p.T + RG - 1) / RG);
  }
  __device__ int kblocks() const { return H / tc::TK; }
  __device__ uint32_t* status() const { return p.status; }
  __device__ unsigned long long* trace() const { return p.trace; }  // slots 0..7
  __device__ void tile(int i, TileInfo& t, const uint8_t* tbl) const {
    const int* mtp = reinterpret_cast<const int*>(tbl);
    const int* off = mtp + (E + 1);
    const int routed = NCT_GU * mtp[E];
    int j;
    if (!shared_tile(i, routed, j)) {
      const int e = GroupTable::find(mtp, NCT_GU, j);
      const int local = j - NCT_GU * mtp[e];
      const int mt = local / NCT_GU, nt = local % NCT_GU;  // column blocks of a row group together
      t.amap = &xs;
      t.a_row0 = off[e] + mt * RG;
      t.b_row0 = e * H;
      t.bmap[0] = &wg;
      t.bmap[1] = &wu;
      t.row0 = off[e] + mt * RG;
      t.valid = min(RG, off[e + 1] - off[e] - mt * RG);
      t.col0 = nt * 64;
      t.aux = 0;
    } else {
      const int ng = (p.T + RG - 1) / RG;
      const int nt = j / ng, g = j % ng;
      t.amap = &xin_c;
      t.a_row0 = g * RG;
      t.b_row0 = 0;
      t.bmap[0] = &wsg;
      t.bmap[1] = &wsu;
      t.row0 = g * RG;
      t.valid = min(RG, p.T - g * RG);
      t.col0 = nt * 64;
      t.aux = 1;
    }
    t.bcol[0] = t.bcol[1] = t.col0;
    t.n = (t.valid + 15) & ~15;
  }
  // h = bf16(silu(gate) * up) into h (routed) or hs (shared).  Per 32-row chunk the gate lanes
  // (0..63) and the up lanes (64..127) swap halves through shared memory -- the up lanes receive
  // the gate of rows 16..31, the gate lanes the up of rows 0..15 -- so all four warps share the
  // work.
  __device__ void epilogue(const TileInfo& t, uint32_t trow, int row, uint8_t* epi, const uint8_t*) const {
    float* xch = reinterpret_cast<float*>(epi);  // [2][16 rows][64 columns] fp32
    const bool gate_lane = row < 64;
    const int f = row & 63;
    const int q0 = gate_lane ? 0 : 16;  // rows of the chunk this lane writes
    float* give = xch + (gate_lane ? 1024 : 0) + f;
    const float* take = xch + (gate_lane ? 0 : 1024) + f;
    const int ld = t.aux ? p.sw : I;
    bf16* dst = (t.aux ? p.hs : p.h) + (size_t)t.row0 * ld + t.col0 + f;
#pragma unroll 1
    for (int c = 0; c * 32 < t.valid; ++c) {
      float v[32];
      tmem_ld32(trow + uint32_t(c * 32), v);
#pragma unroll
      for (int q = 0; q < 16; ++q) give[q * 64] = gate_lane ? v[16 + q] : v[q];
      epi_sync();
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const int r = c * 32 + q0 + q;
        const float other = take[q * 64];
        const float g = gate_lane ? v[q] : other;
        const float u = gate_lane ? other : v[16 + q];
        if (r < t.valid) dst[(size_t)r * ld] = __float2bfloat16_rn(silu_fast(g) * u);
      }
      epi_sync();  // before the next chunk overwrites the exchange buffer
    }
  }
};

// ================================================================ down (routed + shared)
// COLUMNS: 128 output columns on the TMEM lanes and up to RG = 256 rows as N -- a routed
// expert's rows (h, K = 512; epilogue Yb[row][col] = bf16(gate(row) * acc)) or a 256-token
// group of the shared expert (hs, K = 1024; epilogue S[t][col] = acc in fp32) after the routed
// tiles.
struct DownTC {
  static constexpr bool kColumns = true;
  Params p;
  CUtensorMap h, wd, hs, wsd;
  __device__ void prologue(uint8_t* tbl) const { GroupTable::load(p, tbl); }
  __device__ int num_tiles(const uint8_t* tbl) const {
    return NCT_DN * (reinterpret_cast<const int*>(tbl)[E] + (p.T + RG - 1) / RG);
  }
  __device__ int kblocks() const { return I / tc::TK; }
  __device__ uint32_t* status() const { return p.status; }
  __device__ unsigned long long* trace() const { return p.trace ? p.trace + 8 : nullptr; }  // slots 8..15
  __device__ void tile(int i, TileInfo& t, const uint8_t* tbl) const {
    const int* mtp = reinterpret_cast<const int*>(tbl);
    const int* off = mtp + (E + 1);
    const int ng = (p.T + RG - 1) / RG;
    int j;
    if (!shared_tile(i, NCT_DN * mtp[E], j)) {
      const int e = GroupTable::find(mtp, NCT_DN, j);
      const int local = j - NCT_DN * mtp[e];
      const int mt = local / NCT_DN, nt = local % NCT_DN;  // column blocks of a row group together
      t.amap = &h;
      t.a_row0 = off[e] + mt * RG;
      t.b_row0 = e * I;
      t.bmap[0] = t.bmap[1] = &wd;
      t.row0 = off[e] + mt * RG;
      t.valid = min(RG, off[e + 1] - off[e] - mt * RG);
      t.col0 = nt * 128;
      t.aux = e;
    } else {
      const int nt = j / ng, g = j % ng;
      t.amap = &hs;
      t.a_row0 = g * RG;
      t.b_row0 = 0;
      t.bmap[0] = t.bmap[1] = &wsd;
      t.row0 = g * RG;
      t.valid = min(RG, p.T - g * RG);
      t.col0 = nt * 128;
      t.aux = -1;
      t.nkb = p.sw / tc::TK;
    }
    t.bcol[0] = t.col0;
    t.bcol[1] = t.col0 + 64;
    t.n = (t.valid + 15) & ~15;
  }
  __device__ void epilogue(const TileInfo& t, uint32_t trow, int row, uint8_t* epi, const uint8_t*) const {
    if (t.aux < 0 && p.dense) {  // a dense layer's output: y = bf16(acc [+ x])
      const size_t o = (size_t)t.row0 * H + t.col0 + row;
#pragma unroll 1
      for (int c = 0; c * 32 < t.valid; ++c) {
        float v[32];
        tmem_ld32(trow + uint32_t(c * 32), v);
#pragma unroll
        for (int q = 0; q < 32; ++q) {
          if (c * 32 + q >= t.valid) continue;
          const size_t oq = o + (size_t)(c * 32 + q) * H;
          const float r = (p.flags & 2u) ? __bfloat162float(p.x[oq]) : 0.f;  // residual
          p.y[oq] = __float2bfloat16_rn(v[q] + r);
        }
      }
      return;
    }
    if (t.aux < 0) {
      float* dst = p.S + (size_t)t.row0 * H + t.col0 + row;
#pragma unroll 1
      for (int c = 0; c * 32 < t.valid; ++c) {
        float v[32];
        tmem_ld32(trow + uint32_t(c * 32), v);
#pragma unroll
        for (int q = 0; q < 32; ++q)
          if (c * 32 + q < t.valid) dst[(size_t)(c * 32 + q) * H] = v[q];
      }
      return;
    }
    float* gate = reinterpret_cast<float*>(epi);  // gate of each of the tile's rows
#pragma unroll
    for (int k = 0; k < RG / TM; ++k) {
      const int r = row + k * TM;
      gate[r] = r < t.valid ? __ldcg(p.topk_w + __ldcg(p.perm + t.row0 + r)) : 0.f;
    }
    epi_sync();
    bf16* dst = p.Yb + (size_t)t.row0 * H + t.col0 + row;
#pragma unroll 1
    for (int c = 0; c * 32 < t.valid; ++c) {
      float v[32];
      tmem_ld32(trow + uint32_t(c * 32), v);
#pragma unroll
      for (int q = 0; q < 32; ++q)
        if (c * 32 + q < t.valid) dst[(size_t)(c * 32 + q) * H] = __float2bfloat16_rn(v[q] * gate[c * 32 + q]);
    }
    epi_sync();  // the next tile rewrites the gates
  }
};

// ================================================================ combine
// y[t] = bf16(S[t] + sum_j Yb[inv(t, j)] in slot order (+ x[t])), fp32; one CTA per token,
// each thread 8 columns (16-byte loads and stores, coalesced across the CTA).
__global__ void __launch_bounds__(256) combine_kernel(const __grid_constant__ Params p) {
  pdl_launch_dependents();
  pdl_wait();
  const int tok = blockIdx.x;
  const int col = threadIdx.x * 8;
  int rows[K];
#pragma unroll
  for (int k = 0; k < K; ++k) rows[k] = __ldcg(p.inv + tok * K + k);
  float v[8];
  const float4* s4 = reinterpret_cast<const float4*>(p.S + (size_t)tok * H + col);
  const float4 s0 = __ldcs(s4), s1 = __ldcs(s4 + 1);
  v[0] = s0.x, v[1] = s0.y, v[2] = s0.z, v[3] = s0.w, v[4] = s1.x, v[5] = s1.y, v[6] = s1.z, v[7] = s1.w;
  uint4 yk[K];
#pragma unroll
  for (int k = 0; k < K; ++k) {
    if ((unsigned)rows[k] >= (unsigned)(p.T * K)) {
      record_status(p.status, ST_BOUNDS);
      rows[k] = 0;
    }
    yk[k] = __ldcs(reinterpret_cast<const uint4*>(p.Yb + (size_t)rows[k] * H + col));
  }
#pragma unroll
  for (int k = 0; k < K; ++k) {
    float f[8];
    bf16x8_to_f32(yk[k], f);
#pragma unroll
    for (int z = 0; z < 8; ++z) v[z] += f[z];
  }
  if (p.flags & 2u) {
    float f[8];
    bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(p.x + (size_t)tok * H + col)), f);
#pragma unroll
    for (int z = 0; z < 8; ++z) v[z] += f[z];
  }
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 b = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    w[i] = *reinterpret_cast<const uint32_t*>(&b);
  }
  *reinterpret_cast<uint4*>(p.y + (size_t)tok * H + col) = make_uint4(w[0], w[1], w[2], w[3]);
}

}  // namespace pf
}  // namespace flint
