// Prefill-size path of the Flint MoE layer (T > 256 tokens): the contractions are dense enough
// for the tensor cores, so every GEMM-shaped step runs on the tcgen05 engine (tc_gemm.cuh):
//
//   router    [T x 2048] x W_r [2048 x 256]: epilogue = bias, sigmoid, top-6 with the lower
//             index first on ties, renormalised gates, and a per-tile histogram of the choices;
//   scan      one CTA: counts, offsets, per-tile bases of every expert, M-tile prefix;
//   scatter   one CTA per 128-token tile: stable (t, j)-order placement of the pairs into
//             expert-sorted rows (perm / inv) and the gathered input rows xs[row] = x[t];
//   gate/up   grouped over (expert, 128-column pair of gate and up, 128-row tile) plus the shared
//             expert over (128-column pair, token tile): epilogue h = bf16(silu(g) * u);
//   down      grouped over (expert, 256 output columns, 128-row tile): epilogue
//             Y[row] = bf16(gate(row) * acc);
//   shared down + combine  over (256 output columns, token tile): epilogue
//             y[t] = bf16(acc + sum_j Y[inv(t, j)] in slot order (+ x[t])).
// Tiles of one expert's weight column block are numbered consecutively with the row tile
// fastest, so concurrent CTAs share each weight tile through L2.
#pragma once

#include "common.cuh"
#include "tc_gemm.cuh"

namespace flint {
namespace pf {

using tc::TileInfo;
using tc::TM;
using tc::tmem_ld32;
using tc::epi_sync;

constexpr int NCT_GU = I / 128;   // 4 column pairs of a routed expert's gate/up
constexpr int NCT_SGU = IS / 128; // 8 column pairs of the shared gate/up
constexpr int NCT_OUT = H / 256;  // 8 output column blocks of a down projection

struct Maps {
  CUtensorMap xin;  // [T][H], box 64 x 128 (A operand)
  CUtensorMap xs;   // [6 max_T][H], box 64 x 128
  CUtensorMap h;    // [6 max_T][I], box 64 x 128
  CUtensorMap hs;   // [max_T][IS], box 64 x 128
  CUtensorMap wr;   // [H][E], box 64 x 64 (B operand)
  CUtensorMap wg;   // [E H][I], box 64 x 64
  CUtensorMap wu;
  CUtensorMap wd;   // [E I][H], box 64 x 64
  CUtensorMap wsg;  // [H][IS], box 64 x 64
  CUtensorMap wsu;
  CUtensorMap wsd;  // [IS][H], box 64 x 64
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
  Params p;
  CUtensorMap xin, wr;
  __device__ void prologue(uint8_t*) const {}
  __device__ int num_tiles(const uint8_t*) const { return (p.T + TM - 1) / TM; }
  __device__ int kblocks() const { return H / tc::TK; }
  __device__ uint32_t* status() const { return p.status; }
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
  // Thread `row` owns token row0 + row: its 256 logits stream out of TMEM 32 at a time in
  // expert order; a running top-6 keeps the higher score, and on equal scores the expert seen
  // first (the lower index).
  __device__ void epilogue(const TileInfo& t, uint32_t trow, int row, uint8_t* epi, const uint8_t*) const {
    int* hist = reinterpret_cast<int*>(epi);
    hist[row] = 0;
    hist[row + TM] = 0;
    float s6[K];
    int e6[K];
#pragma unroll
    for (int j = 0; j < K; ++j) {
      s6[j] = -1.f;
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
        const float s = 1.0f / (1.0f + expf(-l));
        if (s > s6[K - 1]) {
          s6[K - 1] = s;
          e6[K - 1] = e;
#pragma unroll
          for (int j = K - 1; j > 0; --j) {
            if (s6[j] > s6[j - 1]) {
              const float ts = s6[j];
              s6[j] = s6[j - 1];
              s6[j - 1] = ts;
              const int te = e6[j];
              e6[j] = e6[j - 1];
              e6[j - 1] = te;
            }
          }
        }
      }
    }
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

// ================================================================ scan (one CTA of 256 threads)
// counts, offsets (+ user counts), per-tile relative bases hbase[tile][e] = sum of earlier
// tiles' choices of e, and the M-tile prefix mtp[e] = sum over e' < e of ceil(n_e' / 128).
__global__ void __launch_bounds__(256) scan_kernel(const __grid_constant__ Params p) {
  __shared__ int s_w[2][8];
  pdl_launch_dependents();
  pdl_wait();
  const int e = threadIdx.x, lane = e & 31, warp = e >> 5;
  const int ntiles = (p.T + TM - 1) / TM;
  int run = 0;
  for (int tt = 0; tt < ntiles; ++tt) {
    p.hbase[(size_t)tt * E + e] = run;
    run += __ldcg(p.hist + (size_t)tt * E + e);
  }
  const int c = run;
  const int mt = (c + TM - 1) / TM;
  int ic = c, im = mt;
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
  const int off_e = bc + ic - c;
  p.counts[e] = c;
  p.offsets[e] = off_e;
  p.mtp[e] = bm + im - mt;
  if (p.out_counts) p.out_counts[e] = c;
  if (e == E - 1) {
    p.offsets[E] = off_e + c;
    p.mtp[E] = bm + im;
  }
}

// ================================================================ scatter + gather
// One CTA (256 threads) per 128-token tile: the tile's 768 (t, j) pairs in order get their
// expert-sorted rows (stable), and the input row of each pair is copied to xs[row].
__global__ void __launch_bounds__(256) scatter_kernel(const __grid_constant__ Params p) {
  __shared__ int s_fill[E];
  __shared__ int s_wcnt[8][E];
  __shared__ int s_rows[TM * K];
  pdl_launch_dependents();
  pdl_wait();
  const int tile = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int t0 = tile * TM;
  const int npairs = min(TM, p.T - t0) * K;
  s_fill[tid] = __ldcg(p.offsets + tid) + __ldcg(p.hbase + (size_t)tile * E + tid);
  __syncthreads();
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
      p.perm[row] = t0 * K + pi;
      p.inv[t0 * K + pi] = row;
      s_rows[pi] = row;
    }
    __syncthreads();
    int add = 0;
    for (int w = 0; w < 8; ++w) add += s_wcnt[w][tid];
    s_fill[tid] += add;
    __syncthreads();
  }
  // gather: warp w copies pairs w, w+8, ...; 256 x 16 bytes per row, 8 per lane
  for (int q = warp; q < npairs; q += 8) {
    const uint4* src = reinterpret_cast<const uint4*>(p.xin + (size_t)(t0 + q / K) * H);
    uint4* dst = reinterpret_cast<uint4*>(p.xs + (size_t)s_rows[q] * H);
#pragma unroll
    for (int k = 0; k < H / 8 / 32; ++k) dst[lane + 32 * k] = __ldg(src + lane + 32 * k);
  }
}

// Routing tables of the grouped GEMMs, copied to shared memory by every CTA: mtp[0..E],
// offsets[0..E].
struct GroupTable {
  __device__ static void load(const Params& p, uint8_t* tbl) {
    int* mtp = reinterpret_cast<int*>(tbl);
    int* off = mtp + (E + 1);
    for (int i = threadIdx.x; i <= E; i += blockDim.x) {
      mtp[i] = __ldcg(p.mtp + i);
      off[i] = __ldcg(p.offsets + i);
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

// ================================================================ gate/up (routed + shared)
struct GateUpTC {
  Params p;
  CUtensorMap xs, xin, wg, wu, wsg, wsu;
  __device__ void prologue(uint8_t* tbl) const { GroupTable::load(p, tbl); }
  __device__ int num_tiles(const uint8_t* tbl) const {
    const int* mtp = reinterpret_cast<const int*>(tbl);
    return NCT_GU * mtp[E] + NCT_SGU * ((p.T + TM - 1) / TM);
  }
  __device__ int kblocks() const { return H / tc::TK; }
  __device__ uint32_t* status() const { return p.status; }
  __device__ void tile(int i, TileInfo& t, const uint8_t* tbl) const {
    const int* mtp = reinterpret_cast<const int*>(tbl);
    const int* off = mtp + (E + 1);
    const int routed = NCT_GU * mtp[E];
    int nt, mt;
    if (i < routed) {
      const int e = GroupTable::find(mtp, NCT_GU, i);
      const int mte = mtp[e + 1] - mtp[e];
      const int local = i - NCT_GU * mtp[e];
      nt = local / mte;
      mt = local % mte;
      t.amap = &xs;
      t.a_row0 = off[e] + mt * TM;
      t.b_row0 = e * H;
      t.bmap[0] = t.bmap[1] = &wg;
      t.bmap[2] = t.bmap[3] = &wu;
      t.row0 = off[e] + mt * TM;
      t.valid = min(TM, off[e + 1] - off[e] - mt * TM);
      t.aux = 0;
    } else {
      const int ntt = (p.T + TM - 1) / TM;
      const int j = i - routed;
      nt = j / ntt;
      mt = j % ntt;
      t.amap = &xin;
      t.a_row0 = mt * TM;
      t.b_row0 = 0;
      t.bmap[0] = t.bmap[1] = &wsg;
      t.bmap[2] = t.bmap[3] = &wsu;
      t.row0 = mt * TM;
      t.valid = min(TM, p.T - mt * TM);
      t.aux = 1;
    }
    t.col0 = nt * 128;
    t.bcol[0] = t.bcol[2] = nt * 128;
    t.bcol[1] = t.bcol[3] = nt * 128 + 64;
  }
  // accumulator columns 0..127 = gate, 128..255 = up (of output columns col0 .. col0+127)
  __device__ void epilogue(const TileInfo& t, uint32_t trow, int row, uint8_t*, const uint8_t*) const {
    bf16* dst = t.aux ? p.hs + (size_t)(t.row0 + row) * IS : p.h + (size_t)(t.row0 + row) * I;
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      float g[32], u[32];
      tmem_ld32(trow + uint32_t(c * 32), g);
      tmem_ld32(trow + uint32_t(128 + c * 32), u);
#pragma unroll
      for (int q = 0; q < 32; ++q) g[q] = silu_f32(g[q]) * u[q];
      if (row < t.valid) store_bf16x32(dst + t.col0 + c * 32, g);
    }
  }
};

// ================================================================ routed down
struct DownTC {
  Params p;
  CUtensorMap h, wd;
  __device__ void prologue(uint8_t* tbl) const { GroupTable::load(p, tbl); }
  __device__ int num_tiles(const uint8_t* tbl) const { return NCT_OUT * reinterpret_cast<const int*>(tbl)[E]; }
  __device__ int kblocks() const { return I / tc::TK; }
  __device__ uint32_t* status() const { return p.status; }
  __device__ void tile(int i, TileInfo& t, const uint8_t* tbl) const {
    const int* mtp = reinterpret_cast<const int*>(tbl);
    const int* off = mtp + (E + 1);
    const int e = GroupTable::find(mtp, NCT_OUT, i);
    const int mte = mtp[e + 1] - mtp[e];
    const int local = i - NCT_OUT * mtp[e];
    const int nt = local / mte, mt = local % mte;
    t.amap = &h;
    t.a_row0 = off[e] + mt * TM;
    t.b_row0 = e * I;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      t.bmap[c] = &wd;
      t.bcol[c] = nt * 256 + c * 64;
    }
    t.row0 = off[e] + mt * TM;
    t.valid = min(TM, off[e + 1] - off[e] - mt * TM);
    t.col0 = nt * 256;
    t.aux = e;
  }
  __device__ void epilogue(const TileInfo& t, uint32_t trow, int row, uint8_t*, const uint8_t*) const {
    const bool ok = row < t.valid;
    const float g = ok ? __ldcg(p.topk_w + __ldcg(p.perm + t.row0 + row)) : 0.f;
    bf16* dst = p.Yb + (size_t)(t.row0 + row) * H + t.col0;
#pragma unroll 1
    for (int c = 0; c < 8; ++c) {
      float v[32];
      tmem_ld32(trow + uint32_t(c * 32), v);
#pragma unroll
      for (int q = 0; q < 32; ++q) v[q] *= g;
      if (ok) store_bf16x32(dst + c * 32, v);
    }
  }
};

// ================================================================ shared down + combine
struct SharedDownTC {
  Params p;
  CUtensorMap hs, wsd;
  __device__ void prologue(uint8_t*) const {}
  __device__ int num_tiles(const uint8_t*) const { return NCT_OUT * ((p.T + TM - 1) / TM); }
  __device__ int kblocks() const { return IS / tc::TK; }
  __device__ uint32_t* status() const { return p.status; }
  __device__ void tile(int i, TileInfo& t, const uint8_t*) const {
    const int ntt = (p.T + TM - 1) / TM;
    const int nt = i / ntt, mt = i % ntt;
    t.amap = &hs;
    t.a_row0 = mt * TM;
    t.b_row0 = 0;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      t.bmap[c] = &wsd;
      t.bcol[c] = nt * 256 + c * 64;
    }
    t.row0 = mt * TM;
    t.valid = min(TM, p.T - mt * TM);
    t.col0 = nt * 256;
    t.aux = 0;
  }
  // y[t] = bf16(S + sum_j Y[inv(t, j)] (+ x[t])), fp32, slot order
  __device__ void epilogue(const TileInfo& t, uint32_t trow, int row, uint8_t*, const uint8_t*) const {
    const bool ok = row < t.valid;
    const int tok = t.row0 + row;
    int rows[K];
#pragma unroll
    for (int k = 0; k < K; ++k) rows[k] = ok ? __ldcg(p.inv + tok * K + k) : 0;
    const bool residual = (p.flags & 2u) != 0;
#pragma unroll 1
    for (int c = 0; c < 8; ++c) {
      float v[32];
      tmem_ld32(trow + uint32_t(c * 32), v);
      if (!ok) continue;
      const int col = t.col0 + c * 32;
#pragma unroll
      for (int k = 0; k < K; ++k) {
        const uint4* y4 = reinterpret_cast<const uint4*>(p.Yb + (size_t)rows[k] * H + col);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float f[8];
          bf16x8_to_f32(__ldcg(y4 + q), f);
#pragma unroll
          for (int z = 0; z < 8; ++z) v[q * 8 + z] += f[z];
        }
      }
      if (residual) {
        const uint4* x4 = reinterpret_cast<const uint4*>(p.x + (size_t)tok * H + col);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float f[8];
          bf16x8_to_f32(__ldg(x4 + q), f);
#pragma unroll
          for (int z = 0; z < 8; ++z) v[q * 8 + z] += f[z];
        }
      }
      store_bf16x32(p.y + (size_t)tok * H + col, v);
    }
  }
};

}  // namespace pf
}  // namespace flint
