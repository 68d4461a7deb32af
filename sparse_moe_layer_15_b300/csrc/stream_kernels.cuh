// Streaming (decode-size) path of the Flint MoE layer, T <= STREAM_MAX_T tokens.
//
// At decode sizes the layer is bound by reading weights once: 6 MB per touched expert plus
// 12 MB of shared expert and 1 MB of router.  Each phase therefore flattens its weight
// traffic into a list of equal 32 KB blocks (64 output columns x 128 or 256 rows of one or
// two matrices), gives every CTA of a one-per-SM persistent grid an equal contiguous range
// of blocks, and streams them through a 4-stage TMA pipeline into shared memory, where CUDA
// cores multiply them against the few token rows.  Consecutive blocks of the same output
// columns accumulate in registers; a block range that splits an item across CTAs leaves a
// partial sum, and the last CTA to finish the item (an integer ticket that also records which
// partial slots exist) adds the partials in block order: deterministic, no float atomics.
//
//   stream_k1: router (8-CTA clusters per 4 tokens, W_r slice by one bulk copy, scores summed
//              over the cluster in distributed shared memory), top-6 + renormalisation and
//              the expert permutation (last cluster); the shared expert's gate/up (SiLU-mul
//              fused) in the persistent CTAs, which also prefetch the shared down matrix.
//   stream_k2: routed gate/up (touched experts only, SiLU-mul fused) and the shared down
//              projection; prefetches the touched experts' down matrices into L2 when they fit.
//   stream_k3: routed down projection scaled by the gate; the last item of each 64-column
//              chunk performs the combine y = S + sum_j Y[inv(t, j)] in slot order (+ x).
#pragma once

#include <cooperative_groups.h>

#include "common.cuh"

namespace flint {
namespace cg = cooperative_groups;

constexpr int NTHREADS = 256;
constexpr int NWARPS = NTHREADS / 32;
constexpr int STREAM_MAX_T = 256;
constexpr int NT_MAX = 8;  // token rows per register block (a "token group")
constexpr int NSTAGE = 4;
constexpr int BLK_BYTES = 32768;
constexpr int GU_ROWS = 128;       // gate/up block: 128 rows x 64 columns of gate and of up
constexpr int DN_ROWS = 256;       // down block: 256 rows x 64 columns
constexpr int GU_KB = H / GU_ROWS;   // 16 blocks per gate/up item
constexpr int SD_KB = IS / DN_ROWS;  // 4 blocks per shared-down item
constexpr int DN_KB = I / DN_ROWS;   // 2 blocks per routed-down item
constexpr int GU_NCH = I / 64;       // 8 column chunks of a routed expert's gate/up
constexpr int SGU_NCH = IS / 64;     // 16 column chunks of the shared gate/up
constexpr int OUT_NCH = H / 64;      // 32 column chunks of a down projection

constexpr int RT_TOK = 4;         // tokens per router cluster
constexpr int RT_CL = 8;          // CTAs per router cluster (K split of H)
constexpr int RT_KR = H / RT_CL;  // 256 router rows per CTA (128 KB, one bulk copy pair)

enum Kind : int { KIND_GU = 0, KIND_SGU = 1, KIND_SD = 2, KIND_DN = 3 };

struct StreamMaps {
  CUtensorMap wg;   // w_gate as [E*H][I], box 64 x 128
  CUtensorMap wu;   // w_up   as [E*H][I], box 64 x 128
  CUtensorMap wd;   // w_down as [E*I][H], box 64 x 256
  CUtensorMap wsg;  // [H][IS], box 64 x 128
  CUtensorMap wsu;  // [H][IS], box 64 x 128
  CUtensorMap wsd;  // [IS][H], box 64 x 256
};

// Largest number of token groups (of NT_MAX expert-sorted rows) a call of T tokens can have.
__host__ __device__ constexpr int max_groups(int T) {
  const int pairs = T * K;
  const int u = pairs < E ? pairs : E;
  const int g = (pairs + NT_MAX - 1) / NT_MAX + u;
  return g < pairs ? g : pairs;
}

// ---------------------------------------------------------------- shared-memory layouts
struct SmemST {  // persistent streaming CTA
  static constexpr int stages = 0;                                  // NSTAGE x 32 KB
  static constexpr int xs = stages + NSTAGE * BLK_BYTES;            // [NT_MAX][<=2048] bf16
  static constexpr int red = xs + NT_MAX * H * 2;                   // [8][NT_MAX][128] f32
  static constexpr int out = red + NWARPS * NT_MAX * 128 * 4;       // [NT_MAX][128] f32
  static constexpr int bars = out + NT_MAX * 128 * 4;               // NSTAGE mbarriers
  static constexpr int misc = bars + 8 * NSTAGE;                    // item broadcast, flags
  static constexpr int meta = misc + 128;                           // [4][E+1] int routing copy
  static constexpr int bytes = meta + 4 * (E + 1) * 4;
};
struct SmemRT {  // router CTA + the permutation
  static constexpr int wr = 0;                                      // [256][256] bf16
  static constexpr int xs = wr + RT_KR * E * 2;                     // [RT_TOK][256] f32
  static constexpr int red = xs + RT_TOK * RT_KR * 4;               // [8][RT_TOK][256] f32
  static constexpr int part = red + NWARPS * RT_TOK * E * 4;        // [RT_TOK][256] f32
  static constexpr int scores = part + RT_TOK * E * 4;              // [RT_TOK][256] f32
  static constexpr int bar = scores + RT_TOK * E * 4;
  static constexpr int flag = bar + 16;
  static constexpr int bytes = flag + 16;
  // permutation scratch aliases `red` (used only after the router is done)
  static constexpr int s_cnt = red;                  // [E] int
  static constexpr int s_fill = s_cnt + E * 4;       // [E] int
  static constexpr int s_wcnt = s_fill + E * 4;      // [8][E] int
  static constexpr int s_wsum = s_wcnt + NWARPS * E * 4;  // [3][8] int + totals
};
static_assert(SmemRT::s_wsum + 128 <= SmemRT::part, "permutation scratch must fit in the router buffer");

constexpr int cmax(int a, int b) { return a > b ? a : b; }
constexpr int K1_SMEM = cmax(SmemST::bytes, SmemRT::bytes) + 1024;
constexpr int K23_SMEM = SmemST::bytes + 1024;

__device__ __forceinline__ uint8_t* aligned_smem(uint8_t* raw) {
  uint32_t a = smem_u32(raw);
  uint32_t pad = (1024u - (a & 1023u)) & 1023u;
  return raw + pad;
}

// ---------------------------------------------------------------- tickets
// Arrive after this CTA's global writes with `add` (nblk in the low 8 bits plus one bit per
// partial slot); returns in every thread the counter value after the add when this CTA
// completed the item (low byte == KB), or 0.  The last arriver resets the counter.
__device__ __forceinline__ uint32_t ticket_add(uint32_t* ticket, uint32_t add, uint32_t KB, int* s_word) {
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint32_t now = atomicAdd(ticket, add) + add;
    const bool last = (now & 0xFFu) == KB;
    if (last) atomicExch(ticket, 0u);
    *s_word = last ? int(now) : 0;
  }
  __syncthreads();
  const uint32_t v = uint32_t(*s_word);
  if (v) __threadfence();
  return v;
}

__device__ __forceinline__ bool ticket_last(uint32_t* ticket, uint32_t total, int* s_word) {
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint32_t old = atomicAdd(ticket, 1u);
    const bool last = (old == total - 1);
    if (last) atomicExch(ticket, 0u);
    *s_word = last ? 1 : 0;
  }
  __syncthreads();
  const bool last = *s_word != 0;
  if (last) __threadfence();
  return last;
}

// ---------------------------------------------------------------- work items
struct Item {
  int kind;
  int idx;   // item index within its kind
  int e;     // routed expert, or -1 for the shared expert
  int row0;  // first row: expert-sorted row (routed) or token (shared)
  int nt;    // rows in this token group (1..NT_MAX)
  int c;     // 64-column chunk
  int KB;    // blocks per item
};

// Shared-memory copy of the routing metadata, per touched expert u: expert id, first sorted
// row, row count and first token group (tgp has U+1 entries).
struct Meta {
  const int* e;
  const int* off;
  const int* cnt;
  const int* tgp;
  int U;       // touched experts
  int groups;  // token groups over all touched experts
};

// Copy the routing metadata written by the router kernel into shared memory (all threads).
__device__ Meta load_meta(const Params& p, uint8_t* sm) {
  int* base = reinterpret_cast<int*>(sm + SmemST::meta);
  Meta m;
  m.U = __ldcg(p.n_touched);
  m.groups = __ldcg(p.n_groups);
  int* e = base;
  int* off = base + (E + 1);
  int* cnt = base + 2 * (E + 1);
  int* tgp = base + 3 * (E + 1);
  for (int u = threadIdx.x; u <= m.U; u += NTHREADS) {
    tgp[u] = __ldcg(p.tgp + u);
    if (u < m.U) {
      const int ex = __ldcg(p.touched + u);
      e[u] = ex;
      off[u] = __ldcg(p.offsets + ex);
      cnt[u] = __ldcg(p.counts + ex);
    }
  }
  __syncthreads();
  m.e = e;
  m.off = off;
  m.cnt = cnt;
  m.tgp = tgp;
  return m;
}

// largest u in [0, n) with tgp[u] <= gi
__device__ __forceinline__ int find_group_owner(const int* tgp, int n, int gi) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tgp[mid] <= gi)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

// Item numbering: routed gate/up items are token-group major (gi * 8 + c); routed down items
// are column-chunk major (c * groups + gi), so that each 64-column chunk of the output is a
// contiguous run of blocks; shared items are token-group major.
__device__ Item decode_item(const Params& p, const Meta& m, int kind, int idx) {
  Item it;
  it.kind = kind;
  it.idx = idx;
  if (kind == KIND_GU || kind == KIND_DN) {
    int gi;
    if (kind == KIND_GU) {
      gi = idx / GU_NCH;
      it.c = idx % GU_NCH;
    } else {
      it.c = idx / m.groups;
      gi = idx % m.groups;
    }
    const int u = find_group_owner(m.tgp, m.U, gi);
    const int tg = gi - m.tgp[u];
    it.e = m.e[u];
    it.row0 = m.off[u] + tg * NT_MAX;
    it.nt = min(NT_MAX, m.cnt[u] - tg * NT_MAX);
    it.KB = kind == KIND_GU ? GU_KB : DN_KB;
  } else {
    const int nch = kind == KIND_SGU ? SGU_NCH : OUT_NCH;
    const int tg = idx / nch;
    it.c = idx % nch;
    it.e = -1;
    it.row0 = tg * NT_MAX;
    it.nt = min(NT_MAX, p.T - tg * NT_MAX);
    it.KB = kind == KIND_SGU ? GU_KB : SD_KB;
  }
  return it;
}

// The blocks of one kernel: [0, n_first) of kind k_first, then [n_first, n_total) of k_second.
struct BlockList {
  int k_first, k_second;
  int n_first, n_total;
  int kb_first, kb_second;
};

__device__ __forceinline__ void block_kind(const BlockList& L, int b, int& kind, int& idx, int& kb) {
  if (b < L.n_first) {
    kind = L.k_first;
    idx = b / L.kb_first;
    kb = b % L.kb_first;
  } else {
    kind = L.k_second;
    const int r = b - L.n_first;
    idx = r / L.kb_second;
    kb = r % L.kb_second;
  }
}

__device__ void issue_block(const Params& p, const Meta& m, const StreamMaps& maps, const BlockList& L, int b,
                            uint8_t* stage, uint64_t* bar) {
  int kind, idx, kb;
  block_kind(L, b, kind, idx, kb);
  const Item it = decode_item(p, m, kind, idx);
  mbar_arrive_expect_tx(bar, BLK_BYTES);
  const int x = it.c * 64;
  switch (kind) {
    case KIND_GU:
      tma_load_2d(stage, &maps.wg, x, it.e * H + kb * GU_ROWS, bar);
      tma_load_2d(stage + BLK_BYTES / 2, &maps.wu, x, it.e * H + kb * GU_ROWS, bar);
      break;
    case KIND_SGU:
      tma_load_2d(stage, &maps.wsg, x, kb * GU_ROWS, bar);
      tma_load_2d(stage + BLK_BYTES / 2, &maps.wsu, x, kb * GU_ROWS, bar);
      break;
    case KIND_SD:
      tma_load_2d(stage, &maps.wsd, x, kb * DN_ROWS, bar);
      break;
    default:
      tma_load_2d(stage, &maps.wd, x, it.e * I + kb * DN_ROWS, bar);
      break;
  }
}

// ---------------------------------------------------------------- the per-CTA stream
struct Stream {
  const Params* p;
  const StreamMaps* maps;
  Meta meta;
  BlockList L;
  int g, nctas;  // this CTA and the grid's streaming CTAs
  int b0, nb;    // this CTA's block range
  uint8_t* sm;
  uint64_t* bars;
  int* misc;  // [0..7]: item broadcast; [8..11]: flags
};

// Wait for stage `st` of block number j: thread 0 waits (bounded); the others observe the
// already-completed phase.  Uniform result across the CTA.
__device__ __forceinline__ bool wait_stage(Stream& S, int j) {
  const int st = j % NSTAGE;
  const uint32_t par = uint32_t(j / NSTAGE) & 1u;
  int* ok = S.misc + 8;
  if (threadIdx.x == 0) *ok = mbar_wait_bounded(S.bars + st, par, S.p->status) ? 1 : 0;
  __syncthreads();
  if (!*ok) return false;
  while (!mbar_try_wait(S.bars + st, par)) {
  }
  return true;
}

// acc[t][m][q] += sum over rows r of block `stg` of xs[t][k0 + r] * tile_m[r][ch*8 + q].
// Lane = (row quarter rsub, 16-byte column chunk ch); warps own contiguous row ranges.
template <int NT, int NM, int KR>
__device__ __forceinline__ void mac_block(float (&acc)[NT][NM][8], const bf16* __restrict__ stg,
                                          const bf16* __restrict__ xs, int xlen, int k0) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int rsub = lane >> 3, ch = lane & 7;
  constexpr int RPW = KR / NWARPS;
#pragma unroll 4
  for (int i = 0; i < RPW / 4; ++i) {
    const int r = warp * RPW + i * 4 + rsub;
    float xv[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) xv[t] = __bfloat162float(xs[t * xlen + k0 + r]);
#pragma unroll
    for (int m = 0; m < NM; ++m) {
      const uint4 w = *reinterpret_cast<const uint4*>(stg + (size_t)m * KR * 64 + r * 64 + ch * 8);
      float wf[8];
      bf16x8_to_f32(w, wf);
#pragma unroll
      for (int t = 0; t < NT; ++t)
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[t][m][q] = fmaf(xv[t], wf[q], acc[t][m][q]);
    }
  }
}

// Sum acc over the row lanes (fixed shuffle tree) and the warps (warp order) into out[t][m*64+c].
template <int NT, int NM>
__device__ __forceinline__ void reduce_acc(float (&acc)[NT][NM][8], float* red, float* out) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int rsub = lane >> 3, ch = lane & 7;
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

__device__ __forceinline__ float* partial_slot(const Params& p, const Item& it, int slot) {
  switch (it.kind) {
    case KIND_GU: return p.P_gu + ((size_t)it.idx * GU_KB + slot) * (NT_MAX * 128);
    case KIND_SGU: return p.P_sgu + ((size_t)it.idx * GU_KB + slot) * (NT_MAX * 128);
    case KIND_SD: return p.P_sd + ((size_t)it.idx * SD_KB + slot) * (NT_MAX * 64);
    default: return p.P_dn + ((size_t)it.idx * DN_KB + slot) * (NT_MAX * 64);
  }
}

__device__ __forceinline__ uint32_t* item_ticket(const Params& p, const Item& it) {
  switch (it.kind) {
    case KIND_GU: return p.tk_gu + it.idx;
    case KIND_SGU: return p.tk_sgu + it.idx;
    case KIND_SD: return p.tk_sd + it.idx;
    default: return p.tk_dn + it.idx;
  }
}

// Final values of an item (fp32 sums [nt][ncol] in `vals`, row stride ncol) -> outputs.
__device__ void item_epilogue(const Params& p, const Item& it, const float* vals) {
  const int nt = it.nt, c = it.c;
  if (it.kind == KIND_GU || it.kind == KIND_SGU) {
    bf16* dst = it.kind == KIND_GU ? p.h : p.hs;
    const int ld = it.kind == KIND_GU ? I : IS;
    for (int q = threadIdx.x; q < nt * 64; q += NTHREADS) {
      const int t = q / 64, j = q % 64;
      const float g = vals[t * 128 + j], u = vals[t * 128 + 64 + j];
      dst[(size_t)(it.row0 + t) * ld + c * 64 + j] = __float2bfloat16_rn(silu_f32(g) * u);
    }
  } else if (it.kind == KIND_SD) {
    for (int q = threadIdx.x; q < nt * 64; q += NTHREADS) {
      const int t = q / 64, j = q % 64;
      p.S[(size_t)(it.row0 + t) * H + c * 64 + j] = vals[t * 64 + j];
    }
  } else {  // routed down: rows scaled by their gate
    for (int q = threadIdx.x; q < nt * 64; q += NTHREADS) {
      const int t = q / 64, j = q % 64;
      const int row = it.row0 + t;
      const float g = __ldcg(p.topk_w + __ldcg(p.perm + row));
      p.Y[(size_t)row * H + c * 64 + j] = g * vals[t * 64 + j];
    }
  }
}

// The combine of output columns [64c, 64c + 64): y = S + sum_j Y[inv(t, j)] in slot order (+x).
__device__ void combine_chunk(const Params& p, int c) {
  const bool residual = (p.flags & 2u) != 0;
  for (int q = threadIdx.x; q < p.T * 64; q += NTHREADS) {
    const int t = q / 64, j = q % 64;
    const int col = c * 64 + j;
    float v = __ldcg(p.S + (size_t)t * H + col);
#pragma unroll
    for (int k = 0; k < K; ++k) v += __ldcg(p.Y + (size_t)__ldcg(p.inv + t * K + k) * H + col);
    if (residual) v += __bfloat162float(p.x[(size_t)t * H + col]);
    p.y[(size_t)t * H + col] = __float2bfloat16_rn(v);
  }
}

// The CTA owning block b when N blocks are split evenly over n CTAs (b0(g) = N*g/n).
__device__ __forceinline__ int block_owner(long long b, long long N, int n) {
  return int(((b + 1) * n - 1) / N);
}

// This CTA has written all its routed-down rows of chunk c: arrive; the last of the CTAs
// that cover the chunk's blocks runs the combine of the chunk.
__device__ void arrive_chunk(Stream& S, int c) {
  const long long N = S.L.n_total;
  const long long per_chunk = (long long)S.meta.groups * DN_KB;
  const int g_lo = block_owner(per_chunk * c, N, S.nctas);
  const int g_hi = block_owner(per_chunk * (c + 1) - 1, N, S.nctas);
  uint32_t expect = 0;
  for (int g = g_lo; g <= g_hi; ++g)
    if (N * (g + 1) / S.nctas > N * g / S.nctas) ++expect;
  if (ticket_last(S.p->tk_comb + c, expect, S.misc + 11)) combine_chunk(*S.p, c);
  __syncthreads();
}

// One segment: blocks [kb_start, kb_start + nblk) of item `it`, consumed as CTA blocks
// j .. j + nblk - 1.  Returns false on a device timeout.
template <int NT, int NM, int KR>
__device__ bool run_segment(Stream& S, const Item& it, int kb_start, int nblk, int& j) {
  const Params& p = *S.p;
  bf16* xs = reinterpret_cast<bf16*>(S.sm + SmemST::xs);
  float* red = reinterpret_cast<float*>(S.sm + SmemST::red);
  float* out = reinterpret_cast<float*>(S.sm + SmemST::out);
  // stage the token group's input rows (bf16) for the whole item
  const int xlen = it.kind == KIND_SD ? IS : it.kind == KIND_DN ? I : H;
  const int cpr = xlen / 8;
  for (int q = threadIdx.x; q < NT * cpr; q += NTHREADS) {
    const int t = q / cpr, k8 = q % cpr;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (t < it.nt) {
      const bf16* src;
      if (it.kind == KIND_GU) {
        const int tok = __ldcg(p.perm + it.row0 + t) / K;
        src = p.xin + (size_t)tok * H;
      } else if (it.kind == KIND_SGU) {
        src = p.xin + (size_t)(it.row0 + t) * H;
      } else if (it.kind == KIND_SD) {
        src = p.hs + (size_t)(it.row0 + t) * IS;
      } else {
        src = p.h + (size_t)(it.row0 + t) * I;
      }
      v = __ldcg(reinterpret_cast<const uint4*>(src) + k8);
    }
    *reinterpret_cast<uint4*>(xs + t * xlen + k8 * 8) = v;
  }
  __syncthreads();
  float acc[NT][NM][8];
#pragma unroll
  for (int t = 0; t < NT; ++t)
#pragma unroll
    for (int m = 0; m < NM; ++m)
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[t][m][q] = 0.f;
  for (int q = 0; q < nblk; ++q, ++j) {
    if (!wait_stage(S, j)) return false;
    const int st = j % NSTAGE;
    mac_block<NT, NM, KR>(acc, reinterpret_cast<const bf16*>(S.sm + SmemST::stages + st * BLK_BYTES), xs, xlen,
                          (kb_start + q) * KR);
    __syncthreads();  // every thread is done with this stage
    if (threadIdx.x == 0 && j + NSTAGE < S.nb)
      issue_block(p, S.meta, *S.maps, S.L, S.b0 + j + NSTAGE, S.sm + SmemST::stages + st * BLK_BYTES,
                  S.bars + st);
  }
  reduce_acc<NT, NM>(acc, red, out);
  constexpr int ncol = NM * 64;
  if (kb_start == 0 && nblk == it.KB) {
    item_epilogue(p, it, out);
    __syncthreads();
    return true;
  }
  float* P = partial_slot(p, it, kb_start);
  for (int q = threadIdx.x; q < it.nt * ncol; q += NTHREADS) P[q] = out[q];
  const uint32_t v = ticket_add(item_ticket(p, it), uint32_t(nblk) | (1u << (8 + kb_start)), uint32_t(it.KB),
                                S.misc + 10);
  if (v) {
    // last arriver: add the partial slots in block order
    const uint32_t mask = v >> 8;
    for (int q = threadIdx.x; q < it.nt * ncol; q += NTHREADS) {
      float s = 0.f;
      for (int sl = 0; sl < it.KB; ++sl)
        if (mask & (1u << sl)) s += __ldcg(partial_slot(p, it, sl) + q);
      out[q] = s;
    }
    __syncthreads();
    item_epilogue(p, it, out);
  }
  __syncthreads();
  return true;
}

template <int NM, int KR>
__device__ __forceinline__ bool run_segment_nt(Stream& S, const Item& it, int kb, int nblk, int& j) {
  if (it.nt <= 1) return run_segment<1, NM, KR>(S, it, kb, nblk, j);
  if (it.nt <= 2) return run_segment<2, NM, KR>(S, it, kb, nblk, j);
  if (it.nt <= 4) return run_segment<4, NM, KR>(S, it, kb, nblk, j);
  return run_segment<8, NM, KR>(S, it, kb, nblk, j);
}

// Persistent stream over blocks [0, n_total) of L, split evenly over `nctas` CTAs (this is
// CTA `g`).  All threads of the CTA call it.  `meta` is the shared-memory routing copy
// (unused by shared-expert-only lists).
__device__ void stream_blocks(const Params& p, const Meta& meta, const StreamMaps& maps, const BlockList& L, int g,
                              int nctas, uint8_t* sm) {
  Stream S;
  S.p = &p;
  S.maps = &maps;
  S.meta = meta;
  S.L = L;
  S.g = g;
  S.nctas = nctas;
  S.sm = sm;
  S.bars = reinterpret_cast<uint64_t*>(sm + SmemST::bars);
  S.misc = reinterpret_cast<int*>(sm + SmemST::misc);
  const long long N = L.n_total;
  S.b0 = int(N * g / nctas);
  const int b1 = int(N * (g + 1) / nctas);
  S.nb = b1 - S.b0;
  if (S.nb <= 0) return;
  if (threadIdx.x == 0) {
    for (int s = 0; s < NSTAGE; ++s) mbar_init(S.bars + s, 1);
    fence_mbar_init();
    for (int s = 0; s < NSTAGE && s < S.nb; ++s)
      issue_block(p, S.meta, maps, L, S.b0 + s, sm + SmemST::stages + s * BLK_BYTES, S.bars + s);
  }
  __syncthreads();
  const bool combine = L.k_first == KIND_DN;
  int cur_chunk = -1;
  int j = 0;
  while (j < S.nb) {
    int kind, idx, kb;
    block_kind(L, S.b0 + j, kind, idx, kb);
    const Item it = decode_item(p, S.meta, kind, idx);  // every thread: shared-memory lookups
    if (combine && it.c != cur_chunk) {
      if (cur_chunk >= 0) arrive_chunk(S, cur_chunk);
      cur_chunk = it.c;
    }
    const int nblk = min(it.KB - kb, S.nb - j);
    bool ok;
    if (kind == KIND_GU || kind == KIND_SGU)
      ok = run_segment_nt<2, GU_ROWS>(S, it, kb, nblk, j);
    else
      ok = run_segment_nt<1, DN_ROWS>(S, it, kb, nblk, j);
    if (!ok) return;
  }
  if (combine && cur_chunk >= 0) arrive_chunk(S, cur_chunk);
}

// Spread a bulk L2 prefetch of `bytes` (multiple of 16) at `base` over `nctas` CTAs.
__device__ __forceinline__ void prefetch_share(const void* base, size_t bytes, int g, int nctas) {
  const size_t per = ((bytes / nctas) + 15) & ~size_t(15);
  const size_t a = per * g;
  if (a >= bytes) return;
  size_t n = per < bytes - a ? per : bytes - a;
  const uint8_t* src = static_cast<const uint8_t*>(base) + a;
  while (n) {
    const uint32_t c = n > 65536 ? 65536u : uint32_t(n);
    prefetch_l2_bulk(src, c);
    src += c;
    n -= c;
  }
}

// ================================================================ K1: router + shared gate/up
__device__ void router_cluster(const Params& p, uint8_t* sm, int cl, int rank);
__device__ void permute_small(const Params& p, uint8_t* sm);

__global__ void __cluster_dims__(RT_CL, 1, 1) __launch_bounds__(NTHREADS)
    stream_k1(const __grid_constant__ Params p, const __grid_constant__ StreamMaps maps, int n_router_ctas,
              int n_stream_ctas) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = aligned_smem(smem_raw);
  pdl_launch_dependents();
  if ((int)blockIdx.x < n_router_ctas) {
    router_cluster(p, sm, blockIdx.x / RT_CL, blockIdx.x % RT_CL);
    return;
  }
  const int g = blockIdx.x - n_router_ctas;
  // the shared down matrix is read by the next kernel: start bringing it into L2
  prefetch_share(p.ws_down, (size_t)IS * H * 2, g, n_stream_ctas);
  pdl_wait();
  const int ntg = (p.T + NT_MAX - 1) / NT_MAX;
  BlockList L;
  L.k_first = KIND_SGU;
  L.k_second = KIND_SGU;
  L.kb_first = L.kb_second = GU_KB;
  L.n_first = L.n_total = ntg * SGU_NCH * GU_KB;
  Meta none{};
  stream_blocks(p, none, maps, L, g, n_stream_ctas, sm);
}

__device__ void router_cluster(const Params& p, uint8_t* sm, int cl, int rank) {
  cg::cluster_group cluster = cg::this_cluster();
  bf16* wr = reinterpret_cast<bf16*>(sm + SmemRT::wr);
  float* xs = reinterpret_cast<float*>(sm + SmemRT::xs);
  float* red = reinterpret_cast<float*>(sm + SmemRT::red);
  float* part = reinterpret_cast<float*>(sm + SmemRT::part);
  float* scores = reinterpret_cast<float*>(sm + SmemRT::scores);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + SmemRT::bar);
  int* flag = reinterpret_cast<int*>(sm + SmemRT::flag);
  const int t0 = cl * RT_TOK;
  const int nt = min(RT_TOK, p.T - t0);
  const int k0 = rank * RT_KR;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  // the router rows [k0, k0 + 256) are one contiguous 128 KB range: two bulk copies
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(bar, RT_KR * E * 2);
    const uint8_t* src = reinterpret_cast<const uint8_t*>(p.w_router + (size_t)k0 * E);
    bulk_g2s(wr, src, RT_KR * E, bar);
    bulk_g2s(reinterpret_cast<uint8_t*>(wr) + RT_KR * E, src + RT_KR * E, RT_KR * E, bar);
  }
  pdl_wait();
  // stage the token rows of this K slice (fp32)
  for (int c = threadIdx.x; c < RT_TOK * (RT_KR / 8); c += NTHREADS) {
    const int t = c / (RT_KR / 8), q = c % (RT_KR / 8);
    float f[8];
    if (t < nt) {
      const uint4 v = *reinterpret_cast<const uint4*>(p.xin + (size_t)(t0 + t) * H + k0 + q * 8);
      bf16x8_to_f32(v, f);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) f[i] = 0.f;
    }
    float4* d = reinterpret_cast<float4*>(xs + t * RT_KR + q * 8);
    d[0] = make_float4(f[0], f[1], f[2], f[3]);
    d[1] = make_float4(f[4], f[5], f[6], f[7]);
  }
  if (threadIdx.x == 0) flag[0] = mbar_wait_bounded(bar, 0, p.status) ? 1 : 0;
  __syncthreads();
  const bool have_w = flag[0] != 0;
  if (have_w)
    while (!mbar_try_wait(bar, 0)) {
    }
  // partial logits: lane owns experts 8*lane..8*lane+7, warp owns rows warp, warp+8, ...
  float acc[RT_TOK][8];
#pragma unroll
  for (int t = 0; t < RT_TOK; ++t)
#pragma unroll
    for (int q = 0; q < 8; ++q) acc[t][q] = 0.f;
  if (have_w) {
#pragma unroll 8
    for (int i = 0; i < RT_KR / NWARPS; ++i) {
      const int r = warp + i * NWARPS;
      const uint4 w = *reinterpret_cast<const uint4*>(wr + r * E + lane * 8);
      float wf[8];
      bf16x8_to_f32(w, wf);
#pragma unroll
      for (int t = 0; t < RT_TOK; ++t) {
        const float xv = xs[t * RT_KR + r];
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[t][q] = fmaf(xv, wf[q], acc[t][q]);
      }
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
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (lane + 32 * q == e) key[q] = 0;  // scores are >= 0: an emptied slot never wins
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
  if (!ticket_last(p.tk_router, n_clusters, flag + 1)) return;
  permute_small(p, sm);
}

// Stable counting sort of the T*K (token, slot) pairs by expert, in one CTA; also the list
// of touched experts and the prefix of their token groups.
__device__ void permute_small(const Params& p, uint8_t* sm) {
  int* s_cnt = reinterpret_cast<int*>(sm + SmemRT::s_cnt);
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
  // exclusive scans over experts (tid == expert): counts, touched flags, token groups
  const int c = s_cnt[tid];
  const int f = c > 0 ? 1 : 0;
  const int ng = (c + NT_MAX - 1) / NT_MAX;
  int ic = c, jf = f, kg = ng;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int a = __shfl_up_sync(0xffffffffu, ic, off);
    const int b = __shfl_up_sync(0xffffffffu, jf, off);
    const int d = __shfl_up_sync(0xffffffffu, kg, off);
    if (lane >= off) {
      ic += a;
      jf += b;
      kg += d;
    }
  }
  if (lane == 31) {
    s_wsum[warp] = ic;
    s_wsum[NWARPS + warp] = jf;
    s_wsum[2 * NWARPS + warp] = kg;
  }
  __syncthreads();
  int bc = 0, bf = 0, bg = 0;
  for (int w = 0; w < warp; ++w) {
    bc += s_wsum[w];
    bf += s_wsum[NWARPS + w];
    bg += s_wsum[2 * NWARPS + w];
  }
  const int off_e = bc + ic - c;
  const int pos = bf + jf - f;
  const int gpre = bg + kg - ng;
  s_fill[tid] = off_e;
  p.counts[tid] = c;
  p.offsets[tid] = off_e;
  if (p.out_counts) p.out_counts[tid] = c;
  if (f) {
    p.touched[pos] = tid;
    p.tgp[pos] = gpre;
  }
  if (tid == NTHREADS - 1) {
    p.offsets[E] = off_e + c;
    *p.n_touched = pos + f;
    *p.n_groups = gpre + ng;
    p.tgp[pos + f] = gpre + ng;
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
}

// ================================================================ K2: routed gate/up + shared down
__global__ void __launch_bounds__(NTHREADS)
    stream_k2(const __grid_constant__ Params p, const __grid_constant__ StreamMaps maps) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = aligned_smem(smem_raw);
  pdl_launch_dependents();
  pdl_wait();
  const Meta meta = load_meta(p, sm);
  const int groups = meta.groups;
  const int U = meta.U;
  // the next kernel reads the touched experts' down matrices: prefetch them when they fit
  if ((unsigned long long)U * I * H * 2 <= p.prefetch_bytes_max && threadIdx.x == 0) {
    const size_t per_e = (size_t)I * H * 2;
    const size_t total = per_e * U;
    const size_t share = ((total / gridDim.x) + 15) & ~size_t(15);
    size_t a = share * blockIdx.x, b = a + share < total ? a + share : total;
    while (a < b) {
      const int u = int(a / per_e);
      const size_t in_e = a % per_e;
      size_t n = per_e - in_e;
      if (n > b - a) n = b - a;
      if (n > 65536) n = 65536;
      const int e = __ldcg(p.touched + u);
      prefetch_l2_bulk(reinterpret_cast<const uint8_t*>(p.w_down + (size_t)e * I * H) + in_e, uint32_t(n));
      a += n;
    }
  }
  const int ntg = (p.T + NT_MAX - 1) / NT_MAX;
  BlockList L;
  L.k_first = KIND_GU;
  L.kb_first = GU_KB;
  L.n_first = groups * GU_NCH * GU_KB;
  L.k_second = KIND_SD;
  L.kb_second = SD_KB;
  L.n_total = L.n_first + ntg * OUT_NCH * SD_KB;
  stream_blocks(p, meta, maps, L, blockIdx.x, gridDim.x, sm);
}

// ================================================================ K3: routed down + combine
__global__ void __launch_bounds__(NTHREADS)
    stream_k3(const __grid_constant__ Params p, const __grid_constant__ StreamMaps maps) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = aligned_smem(smem_raw);
  pdl_launch_dependents();
  pdl_wait();
  const Meta meta = load_meta(p, sm);
  BlockList L;
  L.k_first = L.k_second = KIND_DN;
  L.kb_first = L.kb_second = DN_KB;
  L.n_first = L.n_total = meta.groups * OUT_NCH * DN_KB;
  stream_blocks(p, meta, maps, L, blockIdx.x, gridDim.x, sm);
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
  *reinterpret_cast<uint4*>(p.xn + (size_t)t * H + threadIdx.x * 8) =
      make_uint4(packed[0], packed[1], packed[2], packed[3]);
}

}  // namespace flint
