// Decode-size path of the Flint MoE layer (T <= STREAM_MAX_T tokens): ONE persistent
// cooperative kernel per forward.
//
// At these sizes the layer is bound by reading weights once -- 6 MB per touched expert, 12 MB
// of shared expert, 1 MB of router -- and by latency: a separate kernel per step pays a
// launch, a ramp-up and a tail each time.  So one CTA per SM runs every step in turn, the
// steps separated by grid-wide barriers (bounded spins on a global counter; the cooperative
// launch guarantees that all CTAs are resident):
//
//   A  router partial logits (blocks of 64 W_r rows, all 256 experts); the shared down matrix
//      is prefetched into L2;
//   -- barrier --
//   B  routing: logits summed over the 32 row blocks in order, + bias, sigmoid, top-6 with
//      the lower index first on ties, renormalised gates; for T <= 4 every CTA routes every
//      token itself (no barrier), otherwise each CTA routes its own tokens and a barrier
//      publishes them; then every CTA builds the expert permutation (stable counting sort)
//      in its own shared memory;
//   C  routed gate/up (touched experts only) and the shared expert's gate/up, with fused
//      SiLU-mul; the touched experts' down matrices are prefetched into L2 when they fit;
//   -- barrier --
//   D  routed down projection scaled by the gates, and the shared down projection;
//   -- barrier --
//   E  the combine y = S + sum_j Y[inv(t, j)] in slot order (+ x), spread over the grid.
//
// Within a step the weight traffic is a list of equal 32 KB blocks -- 64 rows x 128 output
// columns of gate and of up, 128 rows x 128 output columns of a down matrix, or 64 router
// rows x 256 experts -- and every CTA takes an equal contiguous range.  A producer warp
// streams the range through a 4-stage TMA ring of 128-byte swizzled boxes; a block is read as
// 8 or 16 KB boxes, two adjacent 64-column chunks of the same rows side by side (measured:
// 5.3 TB/s against 4.8-4.9 for one 64-column chunk of twice the rows).  Eight consumer warps
// multiply each block against the current token group (8 rows, or 16 above 64 tokens) with
// warp-level bf16 MMAs (m16n8k16, fp32 accumulate), each warp owning its own output columns
// over all rows of the block, so a block needs no cross-warp reduction.  Blocks of the same
// output columns (one item) accumulate in registers.  A CTA's range splits at most two items,
// one where it starts and one where it ends: each split piece goes to one of the CTA's two
// partial slots, and the last CTA to finish the item (an integer ticket counting its blocks)
// adds the pieces in block order, finding them from the range arithmetic alone:
// deterministic, no floating-point atomics.
#pragma once

#include "common.cuh"

namespace flint {

constexpr int NCONS = 256;               // consumer threads (8 warps)
constexpr int NWARPS = NCONS / 32;
constexpr int NTHREADS = NCONS + 32;     // + one producer warp
constexpr int STREAM_MAX_T = 256;
constexpr int NT_MAX = 16;               // most token rows per group (two 8-token MMA N tiles)
constexpr int NSTAGE = 4;                // measured: 4 stages beat 5 (and 3) over the decode sweep
constexpr int BLK_BYTES = 32768;
constexpr int GU_ROWS = 64;              // gate/up block: 64 rows x 128 columns of gate and of up
constexpr int DN_ROWS = 128;             // down block: 128 rows x 128 columns
constexpr int RT_ROWS = 64;              // router block: 64 rows x 256 experts
constexpr int GU_KB = H / GU_ROWS;       // 32 blocks per gate/up item
constexpr int SD_KB = IS / DN_ROWS;      // 8 blocks per shared-down item
constexpr int DN_KB = I / DN_ROWS;       // 4 blocks per routed-down item
constexpr int RT_NB = H / RT_ROWS;       // 32 router blocks per token group
constexpr int GU_NCB = I / 128;          // 4 column blocks (128 wide) of a routed expert's gate/up
constexpr int SGU_NCB = IS / 128;        // 8 column blocks of the shared gate/up
constexpr int OUT_NCB = H / 128;         // 16 column blocks of a down projection
constexpr int MAX_STREAM_CTAS = 256;     // largest grid of the decode kernel (the workspace holds its partial slots)
constexpr int PSLOT = NT_MAX * 256;      // floats of one partial slot: [rows][256] gate|up, or [rows][128] down
constexpr int REDUNDANT_ROUTING_MAX_T = 4;
constexpr int MAX_PAIRS = STREAM_MAX_T * K;
constexpr int XPAD = 8;                  // bf16 padding of a staged input row (bank spread)

enum Kind : int { KIND_RT = 0, KIND_GU = 1, KIND_SGU = 2, KIND_SD = 3, KIND_DN = 4 };

struct StreamMaps {
  CUtensorMap wr;   // w_router [H][E], box 64 x 64, 128B swizzle
  CUtensorMap wg;   // w_gate as [E*H][I], box 64 x 64 (columns x rows), 128B swizzle
  CUtensorMap wu;   // w_up   as [E*H][I], box 64 x 64
  CUtensorMap wd;   // w_down as [E*I][H], box 64 x 128
  CUtensorMap wsg;  // [H][IS], box 64 x 64
  CUtensorMap wsu;  // [H][IS], box 64 x 64
  CUtensorMap wsd;  // [IS][H], box 64 x 128
};

// NVFP4 expert weights (Params::fp4), kept in the workspace (Params::fp4_maps), K-major: for a
// matrix W [K][N] of y = x W, E2M1 codes [N][K/2] uint8 (two consecutive k per byte) and E4M3
// scales [N][K/16] uint8.  Gate/up codes: 3-D maps (128 bytes of a row, rows, the row's eight
// 128-byte pieces), boxes of 128 x 16 rows x 8 with the 128-byte swizzle (shared-memory line = piece
// x 16 + row, so the rows of an MMA fragment fall on distinct banks); their scales: boxes of 128
// bytes x 16 rows.  Down codes: boxes of 128 bytes x 128 rows (128-byte swizzle); their scales: the
// block's 4 KB as 32 rows of 128 bytes.
struct Fp4Maps {
  CUtensorMap qg, qu, qd, qsg, qsu, qsd;  // codes: [E*I][H/2], ., [E*H][I/2], [IS][H/2], ., [H][IS/2]
  CUtensorMap sg, su, sd, ssg, ssu, ssd;  // scales: [E*I][H/16], ., [E*H][I/16], [IS][H/16], ., [H][IS/16]
};

// Kernel modes, each its own instantiation (the bf16 MoE kernel carries no code of the others:
// its latency-bound phases run cold instruction fetches once per call).
constexpr int MODE_MOE = 0;    // the MoE layer, bf16 weights
constexpr int MODE_FP4 = 1;    // the MoE layer, NVFP4 expert weights
constexpr int MODE_DENSE = 2;  // a dense SwiGLU MLP layer (the shared-expert steps at width ID)

// ---- NVFP4 streaming (decode sizes): a gate/up block is 16 columns x all 2048 k of gate and of up
// (each matrix's 16 K-major rows are one contiguous 16 KB of codes and 2 KB of scales: one copy
// each; the eight warps split K and add their partial sums in shared memory, so an item is one
// block), a down block 128 columns x 512 k (32 KB of codes in two boxes, 4 KB of scales); the
// codes land in the stage ring, the scales in a ring of 4 KB slots beside it.  Each lane builds
// the MMA A fragments of its rows straight from the codes in registers (e2m1 -> f16 by the
// hardware conversion, times the block's e4m3 scale: exact in f16) and the warp runs f16 MMAs
// against the token rows staged in f16; the tensor scale multiplies the finished item in fp32.
// Token groups of 8 rows only (T <= FP4_MAX_T).
constexpr int FP4_MAX_T = 64;
constexpr int FP4_GU_COLS = 16;               // columns of gate and of up per gate/up block (all K)
constexpr int FP4_DN_ROWS = 512;
constexpr int FP4_GU_KB = 1;                  // one block per gate/up item
constexpr int FP4_DN_KB = I / FP4_DN_ROWS;    // 1 block per routed down item
constexpr int FP4_SD_KB = IS / FP4_DN_ROWS;   // 2 blocks per shared down item
constexpr int FP4_CODE_BYTES = 32768;
constexpr int FP4_SCALE_BYTES = 4096;
static_assert(FP4_CODE_BYTES <= BLK_BYTES, "the codes fit a stage");

// Token rows per group for a call of T tokens: 16 when T > 64 (the weights of the shared
// expert, the router and any expert with more than 8 rows are then streamed once per 16 rows
// instead of 8), else 8 (measured faster for the small calls: fewer zero rows staged and
// computed).
__host__ __device__ constexpr int group_rows(int T) { return T > 64 ? NT_MAX : NT_MAX / 2; }
// A dense layer streams all of its weights once per token group, so its groups are 16 rows from
// 33 tokens on.  Measured (us per call, L2 flushed, 8- vs 16-row groups): T = 64 71.7 vs 61.8,
// T = 32 53.1 vs 53.3, T = 16 43.4 vs 52.0.
__host__ __device__ constexpr int group_rows_mode(int T, int mode) {
  return mode == MODE_DENSE ? (T > 32 ? NT_MAX : NT_MAX / 2) : group_rows(T);
}

// Largest number of token groups (of group_rows(T) expert-sorted rows) a call of T tokens can have.
__host__ __device__ constexpr int max_groups(int T) {
  const int pairs = T * K;
  const int u = pairs < E ? pairs : E;
  const int G = group_rows(T);
  const int g = (pairs + G - 1) / G + u;
  return g < pairs ? g : pairs;
}

// Largest numbers of routed and of shared token groups over the calls of 1..Ts tokens (the group
// width changes at 64 tokens, so the largest call is not always the one with the most groups).
__host__ __device__ constexpr int max_groups_upto(int Ts) {
  const int a = max_groups(Ts < 64 ? Ts : 64), b = max_groups(Ts);
  return a > b ? a : b;
}
__host__ __device__ constexpr int max_shared_groups_upto(int Ts) {
  const int s = Ts < 64 ? Ts : 64;
  const int a = (s + group_rows(s) - 1) / group_rows(s), b = (Ts + group_rows(Ts) - 1) / group_rows(Ts);
  return a > b ? a : b;
}

// ---------------------------------------------------------------- shared memory
// The staged input rows and the output tile come last, so that a call launches with only the
// rows its group width needs (fused_smem_bytes): a smaller footprint leaves more of the SM's
// memory to L1.
struct Smem {
  static constexpr int stages = 0;                                 // NSTAGE x 32 KB
  static constexpr int full = stages + NSTAGE * BLK_BYTES;         // NSTAGE mbarriers
  static constexpr int empty = full + 8 * NSTAGE;                  // NSTAGE mbarriers
  static constexpr int misc = empty + 8 * NSTAGE;                  // flags
  static constexpr int plist = misc + 128;                         // [64] int: partial slots of an item
  static constexpr int meta = plist + 256;                         // [4][E+1] int
  static constexpr int perm = meta + 4 * (E + 1) * 4;              // [MAX_PAIRS] uint16
  static constexpr int inv = perm + MAX_PAIRS * 2;                 // [MAX_PAIRS] uint16
  static constexpr int gw = inv + MAX_PAIRS * 2;                   // [MAX_PAIRS] f32
  static constexpr int xs = gw + MAX_PAIRS * 4;                    // [G][H + XPAD] bf16, G <= NT_MAX
  // then the output tile at out_offset(G), f32: [G][256] (gate/up) or [G][128] (down)
  // reuse of `xs` during routing (between the streaming steps)
  static constexpr int scores = xs;                    // [4][E] f32
  static constexpr int s_cnt = xs + 4 * E * 4;         // [E] int
  static constexpr int s_fill = s_cnt + E * 4;         // [E] int
  static constexpr int s_wcnt = s_fill + E * 4;        // [8][E] int
  static constexpr int s_wsum = s_wcnt + NWARPS * E * 4;  // [4][8] int
  static constexpr int s_idx = s_wsum + 128;           // [MAX_PAIRS] int
};
__host__ __device__ constexpr int xs_bytes(int G) { return G * (H + XPAD) * 2; }
__host__ __device__ constexpr int out_offset(int G) { return Smem::xs + xs_bytes(G); }
// Dynamic shared memory of a launch whose token groups have G rows (+ 1 KB for alignment).
__host__ __device__ constexpr int fused_smem_bytes(int G) { return out_offset(G) + G * 256 * 4 + 1024; }
static_assert(Smem::s_idx + MAX_PAIRS * 4 <= Smem::xs + xs_bytes(NT_MAX / 2), "routing scratch must fit in xs");
static_assert(Smem::perm % 16 == 0 && Smem::gw % 16 == 0 && Smem::xs % 16 == 0, "16-byte aligned tables");
constexpr int FUSED_SMEM = fused_smem_bytes(NT_MAX);  // the largest launch
// NVFP4 launches (8-row groups): the scale slots after the output tile.
__host__ __device__ constexpr int fp4_scl_offset() { return (out_offset(NT_MAX / 2) + NT_MAX / 2 * 256 * 4 + 1023) / 1024 * 1024; }
__host__ __device__ constexpr int fp4_red_offset() { return fp4_scl_offset() + NSTAGE * FP4_SCALE_BYTES; }
// (+ the warps' partial sums of a gate/up block: 8 x 256 floats)
__host__ __device__ constexpr int fp4_smem_bytes() { return fp4_red_offset() + NWARPS * 256 * 4 + 1024; }
static_assert(fp4_smem_bytes() <= FUSED_SMEM, "an NVFP4 launch fits the kernel's shared-memory limit");
static_assert(FUSED_SMEM <= 227 * 1024, "shared memory budget");
static_assert(GU_KB <= 64 && SD_KB <= 64 && DN_KB <= 64, "an item's pieces fit the slot list");
// Most blocks of one step (step C: routed and shared gate/up; step D has half as many per group).
constexpr long long MAX_STEP_BLOCKS = (long long)max_groups_upto(STREAM_MAX_T) * GU_NCB * GU_KB +
                                      (long long)max_shared_groups_upto(STREAM_MAX_T) * SGU_NCB * GU_KB;
static_assert(MAX_STEP_BLOCKS * (MAX_STREAM_CTAS + 1) < (1ll << 32), "32-bit range arithmetic");
// a dense layer's step C (the largest of its two steps) stays below the MoE's
static_assert((long long)max_shared_groups_upto(STREAM_MAX_T) * (ID / 128) * GU_KB <= MAX_STEP_BLOCKS,
              "32-bit range arithmetic, dense layer");
static_assert(ID / DN_ROWS <= 64, "a dense down item's pieces fit the slot list");

__device__ __forceinline__ uint8_t* aligned_smem(uint8_t* raw) {
  uint32_t a = smem_u32(raw);
  uint32_t pad = (1024u - (a & 1023u)) & 1023u;
  return raw + pad;
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Barrier among the 256 consumer threads only (the producer warp keeps streaming).
__device__ __forceinline__ void csync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// ---------------------------------------------------------------- warp MMA helpers
// Byte offset of (row r, bf16 column m) in a tile of 128-byte rows written by TMA with the
// 128-byte swizzle (16-byte chunk index XOR row mod 8).
__device__ __forceinline__ uint32_t swz(int r, int m) {
  return uint32_t(r * 128 + ((((m >> 3) ^ r) & 7) << 4) + (m & 7) * 2);
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&a)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&b)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(b[0]), "=r"(b[1]), "=r"(b[2]), "=r"(b[3])
               : "r"(addr));
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// The same with f16 operands (the NVFP4 mode: its dequantised weights are exact f16 values).
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
template <bool F16>
__device__ __forceinline__ void mma_op(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  if constexpr (F16)
    mma_f16(d, a, b0, b1);
  else
    mma_bf16(d, a, b0, b1);
}

// d[h] += A * B_h over `ksteps` (even) k-steps of 16 rows starting at tile row `r0`, where A =
// the 16 columns [m0, m0+16) of a swizzled weight tile (rows = k) and B_h = the staged input
// rows xs[8h + n][k0 + ...] (8 tokens each, row stride xstride bf16); B_1 (tokens 8..15) only
// when TWO.  Two k-steps per B load.
template <bool TWO, bool F16 = false>
__device__ __forceinline__ void mma_tile_t(float (&d)[2][4], uint32_t tile, int m0, int r0, int ksteps, uint32_t xs,
                                           int xstride, int k0) {
  const int lane = threadIdx.x & 31;
  const int q = lane >> 3, i = lane & 7;
  // A: matrix q -> (m + 8 * (q & 1), k + 8 * (q >> 1)), lane row i
  const int am = m0 + ((q & 1) << 3);
  const int ak = (q >> 1) << 3;
  // B: matrix q -> k offset 8q, lane row = token i (+ 8 for B_1)
  const uint32_t bbase = xs + uint32_t((i * xstride + k0 + q * 8) * 2);
  const uint32_t bhi = uint32_t(8 * xstride * 2);
#pragma unroll 2
  for (int s = 0; s < ksteps; s += 2) {
    uint32_t b[4], b2[4];
    ldsm_x4(bbase + uint32_t(s * 16 * 2), b);
    if constexpr (TWO) ldsm_x4(bbase + bhi + uint32_t(s * 16 * 2), b2);
    uint32_t a[4];
    ldsm_x4_trans(tile + swz(r0 + s * 16 + ak + i, am), a);
    mma_op<F16>(d[0], a, b[0], b[1]);
    if constexpr (TWO) mma_op<F16>(d[1], a, b2[0], b2[1]);
    ldsm_x4_trans(tile + swz(r0 + (s + 1) * 16 + ak + i, am), a);
    mma_op<F16>(d[0], a, b[2], b[3]);
    if constexpr (TWO) mma_op<F16>(d[1], a, b2[2], b2[3]);
  }
}

// `two` is warp-uniform: a group of at most 8 rows runs the one-tile loop.
template <bool F16 = false>
__device__ __forceinline__ void mma_tile(float (&d)[2][4], uint32_t tile, int m0, int r0, int ksteps, uint32_t xs,
                                         int xstride, int k0, bool two) {
  if (two)
    mma_tile_t<true, F16>(d, tile, m0, r0, ksteps, xs, xstride, k0);
  else
    mma_tile_t<false, F16>(d, tile, m0, r0, ksteps, xs, xstride, k0);
}

// d[m][h] += A_m * B_h for the two 16-column tiles A_0 = columns [m0, m0+16) and A_1 =
// [m0+16, m0+32) of a swizzled weight tile (rows 0 .. 16*ksteps-1 = k), B_h as in mma_tile_t;
// one B load feeds both tiles.
template <bool TWO, bool F16 = false>
__device__ __forceinline__ void mma_pair_t(float (&d)[2][2][4], uint32_t tile, int m0, int ksteps, uint32_t xs,
                                           int xstride, int k0) {
  const int lane = threadIdx.x & 31;
  const int q = lane >> 3, i = lane & 7;
  const int am = m0 + ((q & 1) << 3);
  const int ak = (q >> 1) << 3;
  const uint32_t bbase = xs + uint32_t((i * xstride + k0 + q * 8) * 2);
  const uint32_t bhi = uint32_t(8 * xstride * 2);
#pragma unroll
  for (int s = 0; s < ksteps; s += 2) {
    uint32_t b[4], b2[4];
    ldsm_x4(bbase + uint32_t(s * 16 * 2), b);
    if constexpr (TWO) ldsm_x4(bbase + bhi + uint32_t(s * 16 * 2), b2);
#pragma unroll
    for (int m = 0; m < 2; ++m) {
      uint32_t a[4];
      ldsm_x4_trans(tile + swz(s * 16 + ak + i, am + 16 * m), a);
      mma_op<F16>(d[m][0], a, b[0], b[1]);
      if constexpr (TWO) mma_op<F16>(d[m][1], a, b2[0], b2[1]);
      ldsm_x4_trans(tile + swz((s + 1) * 16 + ak + i, am + 16 * m), a);
      mma_op<F16>(d[m][0], a, b[2], b[3]);
      if constexpr (TWO) mma_op<F16>(d[m][1], a, b2[2], b2[3]);
    }
  }
}

template <bool F16 = false>
__device__ __forceinline__ void mma_pair(float (&d)[2][2][4], uint32_t tile, int m0, int ksteps, uint32_t xs,
                                         int xstride, int k0, bool two) {
  if (two)
    mma_pair_t<true, F16>(d, tile, m0, ksteps, xs, xstride, k0);
  else
    mma_pair_t<false, F16>(d, tile, m0, ksteps, xs, xstride, k0);
}

// ---------------------------------------------------------------- tickets and barriers
// Arrive (consumers) after this CTA's global writes, adding the `nblk` blocks of the item that
// this CTA computed; true in every consumer thread when this CTA completed the item (the count
// reached KB).  The last arriver resets the counter.
__device__ __forceinline__ bool ticket_add(uint32_t* ticket, uint32_t nblk, uint32_t KB, int* s_word) {
  __threadfence();
  csync();
  if (threadIdx.x == 0) {
    const uint32_t now = atomicAdd(ticket, nblk) + nblk;
    const bool last = now == KB;
    if (last) atomicExch(ticket, 0u);
    *s_word = last ? 1 : 0;
  }
  csync();
  const bool last = *s_word != 0;
  if (last) __threadfence();
  return last;
}

// `all_threads`: synchronise the whole CTA (else the consumers only).
__device__ __forceinline__ bool ticket_last(uint32_t* ticket, uint32_t total, int* s_word, bool all_threads) {
  __threadfence();
  if (all_threads)
    __syncthreads();
  else
    csync();
  if (threadIdx.x == 0) {
    const uint32_t old = atomicAdd(ticket, 1u);
    const bool last = (old == total - 1);
    if (last) atomicExch(ticket, 0u);
    *s_word = last ? 1 : 0;
  }
  if (all_threads)
    __syncthreads();
  else
    csync();
  const bool last = *s_word != 0;
  if (last) __threadfence();
  return last;
}

// Grid-wide barrier number `k` (1, 2, ...) of this forward: every CTA adds 1 to a global
// counter and waits (bounded) until it reaches k * gridDim.x.  Returns false on timeout.
__device__ bool grid_sync(const Params& p, int k, int* s_flag) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(p.bar_count, 1u);
    const uint32_t target = uint32_t(k) * gridDim.x;
    int ok = 1;
    if (ld_acquire_u32(p.bar_count) < target) {
      const uint64_t t0 = globaltimer_ns();
      while (ld_acquire_u32(p.bar_count) < target) {
        if (globaltimer_ns() - t0 > WAIT_LIMIT_NS) {
          record_status(p.status, ST_TIMEOUT);
          ok = 0;
          break;
        }
      }
    }
    __threadfence();
    *s_flag = ok;
  }
  __syncthreads();
  return *s_flag != 0;
}

// After the last barrier: the last CTA to get here resets the barrier counter and the first
// `ng` routed and `ns` shared token-group counters of the dataflow (every CTA is done with them).
__device__ void grid_done(const Params& p, int* s_flag, int ng = 0, int ns = 0) {
  if (!ticket_last(p.bar_done, gridDim.x, s_flag, true)) return;
  if (threadIdx.x == 0) atomicExch(p.bar_count, 0u);
  for (int i = threadIdx.x; i < ng; i += blockDim.x) p.hdone[i] = 0u;
  for (int i = threadIdx.x; i < ns; i += blockDim.x) p.hsdone[i] = 0u;
}

// Wait for an mbarrier phase; on running out of time record ST_TIMEOUT and go on (the
// results are then garbage, flagged by the status word, and nothing hangs).
__device__ __forceinline__ void mbar_wait_or_flag(uint64_t* bar, uint32_t parity, uint32_t* status) {
  if (mbar_try_wait(bar, parity)) return;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > WAIT_LIMIT_NS) {
      record_status(status, ST_TIMEOUT);
      return;
    }
  }
}

// ---------------------------------------------------------------- work items
struct Item {
  int kind;
  int idx;   // item index within its kind
  int e;     // routed expert, or -1
  int row0;  // first row: expert-sorted row (routed), token (shared / router)
  int nt;    // rows in this token group (1..NT_MAX)
  int c;     // 128-column block (router: row block)
  int KB;    // blocks per item
};

// Shared-memory routing tables of this CTA, per touched expert u: expert id, first sorted
// row, row count, first token group (tgp has U+1 entries).
struct Meta {
  const int* e;
  const int* off;
  const int* cnt;
  const int* tgp;
  int U;
  int groups;
};

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

// Item numbering is token-group major for every kind (router: tg * 32 + row block; routed:
// gi * chunks + c; shared: tg * chunks + c), so that consecutive items of a CTA's range
// usually share their token group and its staged input rows.
// K blocks per item of a kind: 64-row (gate/up) or 128-row (down) bf16 blocks, or the NVFP4
// blocks of 256 / 512 rows.
// Column blocks of a routed and of the shared expert's gate/up, per token group.
template <int MODE>
__host__ __device__ constexpr int gu_ncb() { return MODE == MODE_FP4 ? I / FP4_GU_COLS : GU_NCB; }
template <int MODE>
__host__ __device__ constexpr int sgu_ncb() {
  return MODE == MODE_FP4 ? IS / FP4_GU_COLS : MODE == MODE_DENSE ? ID / 128 : SGU_NCB;
}

template <int MODE>
__device__ __forceinline__ int kblocks_of(const Params& p, int kind) {
  switch (kind) {
    case KIND_RT: return 1;
    case KIND_GU:
    case KIND_SGU: return MODE == MODE_FP4 ? FP4_GU_KB : GU_KB;
    case KIND_DN: return MODE == MODE_FP4 ? FP4_DN_KB : DN_KB;
    default: return MODE == MODE_FP4 ? FP4_SD_KB : MODE == MODE_DENSE ? ID / DN_ROWS : SD_KB;
  }
}

template <int MODE>
__device__ __forceinline__ Item decode_item(const Params& p, const Meta& m, int kind, int idx) {
  const int T = p.T;
  const int sncb = sgu_ncb<MODE>();  // column blocks of the shared gate/up
  Item it;
  it.kind = kind;
  it.idx = idx;
  if (kind == KIND_GU || kind == KIND_DN) {
    const int nch = kind == KIND_GU ? gu_ncb<MODE>() : OUT_NCB;
    const int gi = idx / nch;
    it.c = idx % nch;
    const int u = find_group_owner(m.tgp, m.U, gi);
    const int tg = gi - m.tgp[u];
    const int G = group_rows_mode(T, MODE);
    it.e = m.e[u];
    it.row0 = m.off[u] + tg * G;
    it.nt = min(G, m.cnt[u] - tg * G);
    it.KB = kblocks_of<MODE>(p, kind);
  } else {
    const int nch = kind == KIND_RT ? RT_NB : kind == KIND_SGU ? sncb : OUT_NCB;
    const int tg = idx / nch;
    it.c = idx % nch;
    const int G = group_rows_mode(T, MODE);
    it.e = -1;
    it.row0 = tg * G;
    it.nt = min(G, T - tg * G);
    it.KB = kblocks_of<MODE>(p, kind);
  }
  return it;
}

// The blocks of one step: [0, n_first) of kind k_first, then [n_first, n_total) of k_second.
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

// NVFP4 block (codes into `stage`, scales into `scl`), K-major: gate/up 16 columns x all 2048 k of
// gate and of up (a 16 KB code box and a 2 KB scale box each); down 128 columns x 512 k (two 16 KB
// code boxes of 256 k, one 4 KB scale box).
__device__ void issue_block_fp4(const Item& it, const Fp4Maps& maps, int kb, uint8_t* stage, uint8_t* scl,
                                uint64_t* bar) {
  mbar_arrive_expect_tx(bar, FP4_CODE_BYTES + FP4_SCALE_BYTES);
  constexpr int HALF = FP4_CODE_BYTES / 2, SH = FP4_SCALE_BYTES / 2;
  switch (it.kind) {
    case KIND_GU: {
      const int y = it.e * I + it.c * FP4_GU_COLS;
      tma_load_3d(stage, &maps.qg, 0, y, 0, bar);
      tma_load_3d(stage + HALF, &maps.qu, 0, y, 0, bar);
      tma_load_2d(scl, &maps.sg, 0, y, bar);
      tma_load_2d(scl + SH, &maps.su, 0, y, bar);
      break;
    }
    case KIND_SGU: {
      const int y = it.c * FP4_GU_COLS;
      tma_load_3d(stage, &maps.qsg, 0, y, 0, bar);
      tma_load_3d(stage + HALF, &maps.qsu, 0, y, 0, bar);
      tma_load_2d(scl, &maps.ssg, 0, y, bar);
      tma_load_2d(scl + SH, &maps.ssu, 0, y, bar);
      break;
    }
    case KIND_SD: {
      const int y = it.c * 128, x = kb * FP4_DN_ROWS / 2;
      tma_load_2d(stage, &maps.qsd, x, y, bar);
      tma_load_2d(stage + HALF, &maps.qsd, x + 128, y, bar);
      tma_load_2d(scl, &maps.ssd, kb * FP4_DN_ROWS / 16, y, bar);
      break;
    }
    default: {
      const int y = it.e * H + it.c * 128;
      tma_load_2d(stage, &maps.qd, 0, y, bar);
      tma_load_2d(stage + HALF, &maps.qd, 128, y, bar);
      tma_load_2d(scl, &maps.sd, 0, y / 4, bar);  // the block's 128 rows x 32 bytes as 32 x 128
      break;
    }
  }
}

// Issue K block kb of item `it` into a stage.
template <int MODE>
__device__ void issue_block(const Params& p, const StreamMaps& maps, const Item& it, int kb, uint8_t* stage,
                            uint64_t* bar, uint8_t* scl) {
  const int kind = it.kind;
  if (MODE == MODE_FP4 && kind != KIND_RT) {
    issue_block_fp4(it, *static_cast<const Fp4Maps*>(p.fp4_maps), kb, stage, scl, bar);
    return;
  }
  mbar_arrive_expect_tx(bar, BLK_BYTES);
  // gate/up: boxes [gate chunk 2c | gate 2c+1 | up 2c | up 2c+1] of 8 KB; down: [chunk 2c | 2c+1]
  // of 16 KB (64 columns each: the 128-byte swizzle span)
  const int x = it.c * 128;
  constexpr int Q = BLK_BYTES / 4, Hb = BLK_BYTES / 2;
  switch (kind) {
    case KIND_RT:
#pragma unroll
      for (int q = 0; q < 4; ++q) tma_load_2d(stage + q * Q, &maps.wr, q * 64, it.c * RT_ROWS, bar);
      break;
    case KIND_GU: {
      const int y = it.e * H + kb * GU_ROWS;
      tma_load_2d(stage, &maps.wg, x, y, bar);
      tma_load_2d(stage + Q, &maps.wg, x + 64, y, bar);
      tma_load_2d(stage + 2 * Q, &maps.wu, x, y, bar);
      tma_load_2d(stage + 3 * Q, &maps.wu, x + 64, y, bar);
      break;
    }
    case KIND_SGU: {
      const int y = kb * GU_ROWS;
      tma_load_2d(stage, &maps.wsg, x, y, bar);
      tma_load_2d(stage + Q, &maps.wsg, x + 64, y, bar);
      tma_load_2d(stage + 2 * Q, &maps.wsu, x, y, bar);
      tma_load_2d(stage + 3 * Q, &maps.wsu, x + 64, y, bar);
      break;
    }
    case KIND_SD:
      tma_load_2d(stage, &maps.wsd, x, kb * DN_ROWS, bar);
      tma_load_2d(stage + Hb, &maps.wsd, x + 64, kb * DN_ROWS, bar);
      break;
    default:
      tma_load_2d(stage, &maps.wd, x, it.e * I + kb * DN_ROWS, bar);
      tma_load_2d(stage + Hb, &maps.wd, x + 64, it.e * I + kb * DN_ROWS, bar);
      break;
  }
}

// ---------------------------------------------------------------- the per-CTA stream
struct Stream {
  const Params* p;
  const StreamMaps* maps;
  Meta meta;
  BlockList L;
  int nctas;
  int b0, nb;      // this CTA's block range in the current step
  int ring;        // blocks streamed by this CTA before this step (ring position)
  int first_slot;  // trace slot stamped when the step's first block has arrived
  int x_cls, x_row0, x_k0;  // what the staged input rows hold (-1: nothing valid), from column x_k0
  uint8_t* sm;
  uint64_t* full;
  uint64_t* empty;
  int* misc;  // [8..15]: flags
  int* plist;  // partial slots of the item being finished
  float* out;  // output tile of the current segment
  int comb_items;  // > 0: combine each 128-column block when its comb_items down items are done
  bool dataflow;   // gate/up items signal their token group; down items wait for theirs (no C-D barrier)
  uint32_t* sig_ctr;  // the token-group counter with finished items not yet signalled (dataflow)
  uint32_t sig_n;     // how many
  float* pbank;    // the current step's partial slots (steps C and D use separate banks)
  const uint16_t* perm;
  const uint16_t* inv;
  const float* gw;
};

__device__ __forceinline__ uint8_t* stage_ptr(const Stream& S, int j) {
  return S.sm + Smem::stages + ((S.ring + j) % NSTAGE) * BLK_BYTES;
}

// Producer (one lane): issue blocks [from, to) of this CTA's range of the step into the stage ring.
template <int MODE>
__device__ void produce(Stream& S, int from, int to) {
  // The item of the current block is decoded once per item (a search of the group tables and
  // divisions by runtime block counts), not once per block: the single issuing thread must keep
  // ahead of the memory system, which takes a 32 KB block every ~0.7 us per SM.
  int kind, idx, kb, kbn = 0;
  Item it;
  for (int j = from; j < to; ++j) {
    if (j > from && kb + 1 < kbn) {
      ++kb;
    } else {
      const int b = S.b0 + j;
      block_kind(S.L, b, kind, idx, kb);
      kbn = b < S.L.n_first ? S.L.kb_first : S.L.kb_second;
      it = decode_item<MODE>(*S.p, S.meta, kind, idx);
    }
    const int pos = S.ring + j;
    const int st = pos % NSTAGE;
    const int use = pos / NSTAGE;
    if (use > 0) mbar_wait_or_flag(S.empty + st, uint32_t(use - 1) & 1u, S.p->status);
    issue_block<MODE>(*S.p, *S.maps, it, kb, S.sm + Smem::stages + st * BLK_BYTES, S.full + st,
                      S.sm + fp4_scl_offset() + st * FP4_SCALE_BYTES);
  }
}

// Consumer side of block j: wait until it has landed.
__device__ __forceinline__ void wait_full(Stream& S, int j) {
  const int pos = S.ring + j;
  mbar_wait_or_flag(S.full + pos % NSTAGE, uint32_t(pos / NSTAGE) & 1u, S.p->status);
  if (j == 0) trace_point(*S.p, S.first_slot);
}

// ---- NVFP4 dequantisation (warp-local: each warp writes exactly the part of the bf16 tile that
// its own MMAs read, so only __syncwarp orders the two)
// Two E2M1 codes (one byte, the first in the low nibble) -> f16x2 (the first in the low half).
__device__ __forceinline__ uint32_t e2m1x2_f16x2(uint32_t byte) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(r) : "r"(byte));
  return r;
}
// Two E4M3 values (the first in the low byte) -> f16x2.
__device__ __forceinline__ uint32_t e4m3x2_f16x2(uint32_t half) {
  uint32_t r;
  asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}" : "=r"(r) : "r"(half));
  return r;
}
// The e4m3 scale bytes k, k + 1 (k even) of 16 bytes (a uint4) as f16x2 (k in the low half).
__device__ __forceinline__ uint32_t scale_pair(const uint4& s, int k) {
  const uint32_t w = k < 4 ? s.x : k < 8 ? s.y : k < 12 ? s.z : s.w;
  return e4m3x2_f16x2((w >> (8 * (k & 3))) & 0xFFFFu);
}
// f16x2 of the low (lo = true) or high half of v in both halves.
__device__ __forceinline__ uint32_t bcast_half(uint32_t v, bool lo) { return __byte_perm(v, 0u, lo ? 0x1010 : 0x3232); }

// Two k-steps (ks, ks + 1) of one 16-row MMA tile of a K-major NVFP4 code tile: `c0` and `c1` are the
// 16 code bytes of rows g and g + 8 for the two k-steps (bytes 0-7: k-step ks, 8-15: ks + 1; in a
// k-step, byte j holds k = 2j, 2j + 1), `sg`, `sg8` the rows' two scales as f16x2.  Lane (g, t)
// takes bytes t and t + 4 of each k-step (the m16n8k16 A layout: k = 2t, 2t + 1 and 2t + 8, 2t + 9),
// converts them to f16 pairs, multiplies by the scale (exact) and runs the MMA against b.
__device__ __forceinline__ void fp4_mma2(float (&d)[4], const uint4& c0, const uint4& c1, uint32_t sg, uint32_t sg8,
                                         int sh, const uint32_t (&b)[4]) {
#pragma unroll
  for (int kk = 0; kk < 2; ++kk) {
    const uint32_t w[4] = {kk ? c0.z : c0.x, kk ? c1.z : c1.x, kk ? c0.w : c0.y, kk ? c1.w : c1.y};
    const uint32_t s0 = bcast_half(sg, kk == 0), s8 = bcast_half(sg8, kk == 0);
    uint32_t a[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t h = e2m1x2_f16x2((w[q] >> sh) & 0xFFu);
      const uint32_t sc = (q & 1) ? s8 : s0;
      const __half2 prod = __hmul2(*reinterpret_cast<const __half2*>(&h), *reinterpret_cast<const __half2*>(&sc));
      a[q] = *reinterpret_cast<const uint32_t*>(&prod);
    }
    mma_f16(d, a, b[2 * kk], b[2 * kk + 1]);
  }
}

// B fragments (m16n8k16) of two k-steps from the staged token rows (f16), as in mma_tile_t.
__device__ __forceinline__ void frag_b2(uint32_t xs, int xstride, int k0, uint32_t (&b)[4]) {
  const int lane = threadIdx.x & 31;
  ldsm_x4(xs + uint32_t(((lane & 7) * xstride + k0 + (lane >> 3) * 8) * 2), b);
}

// Gate/up block (NVFP4): warp w takes the block's k in [256 w, +256) (code piece w) for its 16
// gate and 16 up columns; d[0] = gate, d[1] = up (partial sums over the warp's k).  Codes in
// shared memory: [piece 8][row 16][128 bytes] per matrix (128-byte swizzled lines: both rows of
// a lane, g and g + 8, have the swizzle key g); scales [row 16][128 bytes].
__device__ __forceinline__ void fp4_gateup_block(float (&d)[2][4], const uint8_t* codes, const uint8_t* scl,
                                                 uint32_t xs, int xstride) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, sh = 8 * (lane & 3);
  const uint8_t* row = codes + (warp * FP4_GU_COLS + g) * 128;  // gate, row g of piece `warp`
  uint4 sr[2][2];  // the lane's scale bytes of the warp's k: matrices x rows g, g + 8
#pragma unroll
  for (int m = 0; m < 2; ++m) {
    const uint8_t* sm = scl + m * (FP4_SCALE_BYTES / 2) + 16 * warp;
    sr[m][0] = *reinterpret_cast<const uint4*>(sm + g * 128);
    sr[m][1] = *reinterpret_cast<const uint4*>(sm + (g + 8) * 128);
  }
#pragma unroll
  for (int ks = 0; ks < 16; ks += 2) {  // a 16-byte chunk of each row: k-steps ks, ks + 1
    uint32_t b[4];
    frag_b2(xs, xstride, 256 * warp + ks * 16, b);
    const int off = ((ks >> 1) ^ g) << 4;  // the swizzled chunk (key g: lines g and g + 8)
#pragma unroll
    for (int m = 0; m < 2; ++m) {
      const uint8_t* rm = row + m * (FP4_CODE_BYTES / 2);
      const uint4 c0 = *reinterpret_cast<const uint4*>(rm + off);
      const uint4 c1 = *reinterpret_cast<const uint4*>(rm + 8 * 128 + off);
      fp4_mma2(d[m], c0, c1, scale_pair(sr[m][0], ks), scale_pair(sr[m][1], ks), sh, b);
    }
  }
}

// Down block (NVFP4): warp w takes columns [16 w, +16) over the block's 512 k (two code boxes of
// [128 rows][128 bytes], 128-byte swizzled: rows 16w + g and 16w + g + 8 have the swizzle key g).
__device__ __forceinline__ void fp4_down_block(float (&d)[2][4], const uint8_t* codes, const uint8_t* scl,
                                               uint32_t xs, int xstride, int k0) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, sh = 8 * (lane & 3);
  const int r0 = 16 * warp;
  uint4 sr[2][2];  // the lane's scale rows (32 bytes each): rows g, g + 8 x k halves
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    sr[0][h] = *reinterpret_cast<const uint4*>(scl + (r0 + g) * 32 + 16 * h);
    sr[1][h] = *reinterpret_cast<const uint4*>(scl + (r0 + g + 8) * 32 + 16 * h);
  }
#pragma unroll
  for (int h = 0; h < 2; ++h) {  // code box h: k [256 h, +256)
    const uint8_t* row = codes + h * (FP4_CODE_BYTES / 2) + (r0 + g) * 128;
#pragma unroll
    for (int ks = 0; ks < 16; ks += 2) {
      uint32_t b[4];
      frag_b2(xs, xstride, k0 + h * 256 + ks * 16, b);
      const int off = ((ks >> 1) ^ g) << 4;
      const uint4 c0 = *reinterpret_cast<const uint4*>(row + off);
      const uint4 c1 = *reinterpret_cast<const uint4*>(row + 8 * 128 + off);
      fp4_mma2(d[0], c0, c1, scale_pair(sr[0][h], ks), scale_pair(sr[1][h], ks), sh, b);
    }
  }
}

// Consumer side of block j: this warp is done reading it.
__device__ __forceinline__ void release(Stream& S, int j) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(S.empty + (S.ring + j) % NSTAGE);
}

// Partial slot `slot` (0: the piece that opens CTA `cta`'s range, 1: the piece that closes it) of
// the current step's bank.
__device__ __forceinline__ float* partial_slot(const Stream& S, int cta, int slot) {
  return S.pbank + ((size_t)cta * 2 + slot) * PSLOT;
}

// Partial-slot bank of step C (0) or D (1): without a grid barrier between the two steps a CTA
// may start writing its step-D pieces while another CTA still adds up its step-C ones.
__device__ __forceinline__ float* partial_bank(const Params& p, int bank) {
  return p.P + (size_t)bank * MAX_STREAM_CTAS * 2 * PSLOT;
}

// ---- dataflow between the gate/up and down steps
// The CTA that finishes a gate/up item (its outputs written by all consumers) adds 1 to the
// counter of the item's token group (consumers).
__device__ __forceinline__ void signal_done(uint32_t* ctr) {
  __threadfence();
  csync();
  if (threadIdx.x == 0) atomicAdd(ctr, 1u);
}
// A CTA's finished gate/up items are counted per token group and signalled once per run of
// consecutive items of the group (its items of a group are consecutive in its range), which
// saves a fence and an atomic per item: flush_done signals the pending run, when the CTA starts an
// item of another group or ends the step; pend_done adds one finished item of counter `ctr`.
__device__ __forceinline__ void flush_done(Stream& S) {
  if (S.sig_ctr && S.sig_n) {
    __threadfence();
    csync();
    if (threadIdx.x == 0) atomicAdd(S.sig_ctr, S.sig_n);
  }
  S.sig_ctr = nullptr;
  S.sig_n = 0;
}
__device__ __forceinline__ void pend_done(Stream& S, uint32_t* ctr) {
  S.sig_ctr = ctr;
  ++S.sig_n;
}

// Wait (thread 0, bounded; then the consumers) until a token group's counter reaches `need`.
__device__ __forceinline__ void wait_done(const Params& p, const uint32_t* ctr, uint32_t need) {
  if (threadIdx.x == 0 && ld_acquire_u32(ctr) < need) {
    const uint64_t t0 = globaltimer_ns();
    while (ld_acquire_u32(ctr) < need) {
      if (globaltimer_ns() - t0 > WAIT_LIMIT_NS) {
        record_status(p.status, ST_TIMEOUT);
        break;
      }
    }
  }
  csync();
}

// First block of CTA c's range when n_total blocks are split over nctas CTAs (32-bit: the
// product stays below 2^32, see MAX_STEP_BLOCKS).
__device__ __forceinline__ int range_begin(int n_total, int nctas, int c) {
  return int(unsigned(n_total) * unsigned(c) / unsigned(nctas));
}

// The partial slots holding the pieces of an item split over several CTAs' ranges: blocks
// [s, s + KB) of the step's list.  Written to `list` in block order (thread 0); returns the count.
__device__ int item_slots(int n_total, int nctas, int s, int KB, int* list) {
  const int e = s + KB;
  int c = int(unsigned(s) * unsigned(nctas) / unsigned(n_total));  // range_begin(c) <= s
  int b1 = range_begin(n_total, nctas, c + 1);
  while (c + 1 < nctas && b1 <= s) {
    ++c;
    b1 = range_begin(n_total, nctas, c + 1);
  }
  int n = 0;
  int b0 = range_begin(n_total, nctas, c);
  while (c < nctas && b0 < e) {
    if (b1 > b0 && b1 > s) list[n++] = c * 2 + (b0 >= s ? 0 : 1);  // (an empty range holds no piece)
    ++c;
    b0 = b1;
    b1 = range_begin(n_total, nctas, c + 1);
  }
  return n;
}

__device__ __forceinline__ uint32_t* item_ticket(const Params& p, const Item& it) {
  switch (it.kind) {
    case KIND_GU: return p.tk_gu + it.idx;
    case KIND_SGU: return p.tk_sgu + it.idx;
    case KIND_SD: return p.tk_sd + it.idx;
    default: return p.tk_dn + it.idx;
  }
}

// Final values of an item (fp32 sums [nt][ncol] in `vals`) -> outputs.
template <int MODE>
__device__ void item_epilogue(Stream& S, const Item& it, const float* vals) {
  const Params& p = *S.p;
  const int nt = it.nt, c0 = it.c * 128;
  if (it.kind == KIND_GU || it.kind == KIND_SGU) {  // vals[t][256]: gate columns, then up columns
    bf16* dst = it.kind == KIND_GU ? p.h : p.hs;
    const int ld = it.kind == KIND_GU ? I : MODE == MODE_DENSE ? ID : IS;
    if constexpr (MODE == MODE_FP4) {  // NVFP4: the matrices' tensor scales; h kept in f16
      const float tg = it.kind == KIND_GU ? __ldg(p.ts_gate + it.e) : p.ts_sgate;
      const float tu = it.kind == KIND_GU ? __ldg(p.ts_up + it.e) : p.ts_sup;
      __half* dh = reinterpret_cast<__half*>(dst);
      const int cf = it.c * FP4_GU_COLS;  // vals [t][32]: 16 gate columns, then 16 up columns
      for (int q = threadIdx.x; q < nt * FP4_GU_COLS; q += NCONS) {
        const int t = q / FP4_GU_COLS, j = q % FP4_GU_COLS;
        const float g = vals[t * 32 + j] * tg, u = vals[t * 32 + FP4_GU_COLS + j] * tu;
        dh[(size_t)(it.row0 + t) * ld + cf + j] = __float2half_rn(silu_f32(g) * u);
      }
    } else {
      for (int q = threadIdx.x; q < nt * 128; q += NCONS) {
        const int t = q >> 7, j = q & 127;
        const float g = vals[t * 256 + j], u = vals[t * 256 + 128 + j];
        dst[(size_t)(it.row0 + t) * ld + c0 + j] = __float2bfloat16_rn(silu_f32(g) * u);
      }
    }
  } else if (it.kind == KIND_SD && MODE == MODE_DENSE) {  // a dense layer's output: y = bf16(vals [+ x])
    for (int q = threadIdx.x; q < nt * 128; q += NCONS) {
      const int t = q >> 7, j = q & 127;
      const size_t o = (size_t)(it.row0 + t) * H + c0 + j;
      float v = vals[q];
      if (p.flags & 2u) v += __bfloat162float(p.x[o]);  // residual
      p.y[o] = __float2bfloat16_rn(v);
    }
  } else if (it.kind == KIND_SD) {  // vals[t][128]
    const float ts = MODE == MODE_FP4 ? p.ts_sdown : 1.0f;
    for (int q = threadIdx.x; q < nt * 128; q += NCONS) {
      const int t = q >> 7, j = q & 127;
      p.S[(size_t)(it.row0 + t) * H + c0 + j] = MODE == MODE_FP4 ? vals[q] * ts : vals[q];
    }
  } else {  // routed down: rows scaled by their gate (and, NVFP4, the matrix's tensor scale)
    const float ts = MODE == MODE_FP4 ? __ldg(p.ts_down + it.e) : 1.0f;
    for (int q = threadIdx.x; q < nt * 128; q += NCONS) {
      const int t = q >> 7, j = q & 127;
      const int row = it.row0 + t;
      p.Y[(size_t)row * H + c0 + j] = MODE == MODE_FP4 ? S.gw[S.perm[row]] * (vals[q] * ts) : S.gw[S.perm[row]] * vals[q];
    }
  }
}

// y[t][col .. col+8) = S + sum_j Y[inv(t, j)] in slot order (+ x), one 16-byte store (returned).
__device__ __forceinline__ uint4 combine8(const Params& p, const uint16_t* inv, int t, int col) {
  float v[8];
  const float4* s4 = reinterpret_cast<const float4*>(p.S + (size_t)t * H + col);
  float4 a = __ldcg(s4), b = __ldcg(s4 + 1);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
#pragma unroll
  for (int k = 0; k < K; ++k) {
    const float4* y4 = reinterpret_cast<const float4*>(p.Y + (size_t)inv[t * K + k] * H + col);
    a = __ldcg(y4);
    b = __ldcg(y4 + 1);
    v[0] += a.x; v[1] += a.y; v[2] += a.z; v[3] += a.w; v[4] += b.x; v[5] += b.y; v[6] += b.z; v[7] += b.w;
  }
  if (p.flags & 2u) {  // residual
    float f[8];
    bf16x8_to_f32(*reinterpret_cast<const uint4*>(p.x + (size_t)t * H + col), f);
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] += f[i];
  }
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 h2 = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    w[i] = *reinterpret_cast<const uint32_t*>(&h2);
  }
  const uint4 out = make_uint4(w[0], w[1], w[2], w[3]);
  *reinterpret_cast<uint4*>(p.y + (size_t)t * H + col) = out;
  return out;
}

// The combine, spread over the grid (all threads), after the last grid barrier.
__device__ void combine_share(const Params& p, const uint16_t* inv) {
  const int n8 = p.T * (H / 8);
  for (int q = blockIdx.x * blockDim.x + threadIdx.x; q < n8; q += gridDim.x * blockDim.x)
    combine8(p, inv, q / (H / 8), (q % (H / 8)) * 8);
}

// The combine of 128-column block cb for all tokens (consumers), by the CTA that finished the
// block's last down item.
__device__ void combine_block(const Params& p, const uint16_t* inv, int cb) {
  for (int q = threadIdx.x; q < p.T * 16; q += NCONS) combine8(p, inv, q >> 4, cb * 128 + (q & 15) * 8);
}

// Stage the token group's input rows (bf16, columns [k0, k0 + xlen), row stride xlen + XPAD; rows
// nt .. G-1 zero) for an item (consumers), unless they are the rows staged last (same source,
// group and columns).  xlen <= H: a longer row (a dense layer's down input, 6144 wide) is staged
// in windows.
template <int MODE>
__device__ void stage_inputs(Stream& S, const Item& it, int xlen, int k0 = 0) {
  // NVFP4: the gate/up inputs are staged as f16 (the router's stay bf16), so the shared gate/up
  // rows are a class of their own
  constexpr bool F16X = MODE == MODE_FP4;
  const int cls = it.kind == KIND_GU ? 1 : it.kind == KIND_SD ? 2 : it.kind == KIND_DN ? 3
                  : (F16X && it.kind == KIND_SGU) ? 4 : 0;
  if (cls == S.x_cls && it.row0 == S.x_row0 && k0 == S.x_k0) return;
  S.x_cls = cls;
  S.x_row0 = it.row0;
  S.x_k0 = k0;
  const Params& p = *S.p;
  if (S.dataflow && it.kind == KIND_DN) wait_done(p, p.hdone + it.idx / OUT_NCB, gu_ncb<MODE>());
  if (S.dataflow && it.kind == KIND_SD) wait_done(p, p.hsdone + it.idx / OUT_NCB, sgu_ncb<MODE>());
  // every copy of the group is in flight at once (cp.async, L2 only): one round trip, where a
  // load-then-store loop would pay one per iteration while the weight stream waits
  bf16* xs = reinterpret_cast<bf16*>(S.sm + Smem::xs);
  const int cpr = xlen / 8;
  const int G = group_rows_mode(p.T, MODE);
  for (int q = threadIdx.x; q < G * cpr; q += NCONS) {
    const int t = q / cpr, k8 = q % cpr;
    const bf16* src = p.xin;  // rows nt .. G-1: zero-filled (the address is not read)
    if (t < it.nt) {
      if (it.kind == KIND_GU)
        src = p.xin + (size_t)(S.perm[it.row0 + t] / K) * H;
      else if (it.kind == KIND_SGU || it.kind == KIND_RT)
        src = p.xin + (size_t)(it.row0 + t) * H;
      else if (it.kind == KIND_SD)
        src = MODE == MODE_DENSE ? p.hs + (size_t)(it.row0 + t) * ID + k0 : p.hs + (size_t)(it.row0 + t) * IS;
      else
        src = p.h + (size_t)(it.row0 + t) * I;
    }
    cp16(xs + t * (xlen + XPAD) + k8 * 8, src + k8 * 8, t < it.nt);
  }
  cp_commit();
  cp_wait<0>();
  if (F16X && (it.kind == KIND_GU || it.kind == KIND_SGU)) {
    // bf16 -> f16 in place (inputs |x| < 65504); each thread converts the copies it made
    for (int q = threadIdx.x; q < it.nt * cpr; q += NCONS) {
      uint4* a = reinterpret_cast<uint4*>(xs + (q / cpr) * (xlen + XPAD) + (q % cpr) * 8);
      float f[8];
      bf16x8_to_f32(*a, f);
      uint32_t w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const __half2 h2 = __floats2half2_rn(f[2 * i], f[2 * i + 1]);
        w[i] = *reinterpret_cast<const uint32_t*>(&h2);
      }
      *a = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
  csync();
}

// Router block (one item): partial logits of the token group over 64 router rows, written
// to RP[row block][token][expert].  Warp w owns experts [32w, 32w + 32) (two 16-row tiles).
template <int MODE>
__device__ void run_router_block(Stream& S, const Item& it, int& j) {
  const Params& p = *S.p;
  stage_inputs<MODE>(S, it, H);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  wait_full(S, j);
  const uint32_t tile = smem_u32(stage_ptr(S, j)) + uint32_t((warp >> 1) * (BLK_BYTES / 4));
  const uint32_t xs = smem_u32(S.sm + Smem::xs);
  float d0[2][4] = {}, d1[2][4] = {};
  const int mbase = (warp & 1) * 32;  // column within the 64-expert sub-tile
  const bool two = it.nt > 8;
  mma_tile(d0, tile, mbase, 0, RT_ROWS / 16, xs, H + XPAD, it.c * RT_ROWS, two);
  mma_tile(d1, tile, mbase + 16, 0, RT_ROWS / 16, xs, H + XPAD, it.c * RT_ROWS, two);
  release(S, j);
  // C fragment: (expert m0 + g [+8], token 8 * half + 2*tig [+1])
  const int g = lane >> 2, tig = lane & 3;
  const int e0 = warp * 32;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int e = e0 + h * 16 + g + ((r >> 1) << 3);
        const int t = 8 * h2 + 2 * tig + (r & 1);
        const float v = h ? d1[h2][r] : d0[h2][r];
        if (t < it.nt) p.RP[((size_t)it.c * STREAM_MAX_T + it.row0 + t) * E + e] = v;
      }
    }
  }
  csync();  // xs is restaged by the next item
  ++j;
}

// One segment: blocks [kb_start, kb_start + nblk) of item `it`, consumed as CTA blocks
// j .. j + nblk - 1 (consumers).
template <int MODE>
__device__ void run_segment(Stream& S, const Item& it, int kb_start, int nblk, int& j) {
  const Params& p = *S.p;
  const bool gu = it.kind == KIND_GU || it.kind == KIND_SGU;
  // the token-group counter of a gate/up item; a pending run of another group is signalled now
  uint32_t* gctr = nullptr;
  if (gu && S.dataflow) {
    gctr = it.kind == KIND_GU ? p.hdone + it.idx / gu_ncb<MODE>() : p.hsdone + it.idx / sgu_ncb<MODE>();
    if (S.sig_ctr != gctr) flush_done(S);
  }
  // a shared down input longer than a staged row (a dense layer) is staged from the segment's
  // first K row, and restaged when the segment runs past the window
  int kw = (MODE == MODE_DENSE && it.kind == KIND_SD) ? kb_start * DN_ROWS : 0;  // first staged K column
  int xlen = it.kind == KIND_SD ? (MODE == MODE_DENSE ? min(ID - kw, H) : IS) : it.kind == KIND_DN ? I : H;
  stage_inputs<MODE>(S, it, xlen, kw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int j0 = j;
  const uint32_t xs = smem_u32(S.sm + Smem::xs);
  const bool two = it.nt > 8;
  float* out = S.out;
  const int ncol = gu ? 256 : 128;
  const int g = lane >> 2, tig = lane & 3;
  // C fragment (m16n8): column (weight) m0 + g (+8 for r >= 2), token 8*h2 + 2*tig (+1 for odd r)
  if (gu) {
    // warp w: box w >> 1 (gate 2c, gate 2c+1, up 2c, up 2c+1), columns [32*(w&1), +32) as two
    // 16-column tiles, all 64 rows; out columns: 64 * box + column
    float d[2][2][4] = {};
    const uint32_t sub = uint32_t((warp >> 1) * (BLK_BYTES / 4));
    const int m0 = (warp & 1) * 32;
    if constexpr (MODE == MODE_FP4) {
      // NVFP4 block (one per item): each warp's k piece, then the sum over the warps in shared
      // memory -> out [t][32] (16 gate columns, then 16 up columns)
      float acc[2][4] = {};
      for (int q = 0; q < nblk; ++q, ++j) {
        wait_full(S, j);
        const uint8_t* codes = stage_ptr(S, j);
        const uint8_t* scl = S.sm + fp4_scl_offset() + ((S.ring + j) % NSTAGE) * FP4_SCALE_BYTES;
        fp4_gateup_block(acc, codes, scl, xs, xlen + XPAD);
        release(S, j);
      }
      float* red = reinterpret_cast<float*>(S.sm + fp4_red_offset());
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int r = 0; r < 4; ++r)
          red[warp * 256 + (2 * tig + (r & 1)) * 32 + 16 * m + g + ((r >> 1) << 3)] = acc[m][r];
      csync();
      float sum = 0.f;
#pragma unroll
      for (int w = 0; w < NWARPS; ++w) sum += red[w * 256 + threadIdx.x];
      out[threadIdx.x] = sum;
    } else {
      for (int q = 0; q < nblk; ++q, ++j) {
        wait_full(S, j);
        mma_pair(d, smem_u32(stage_ptr(S, j)) + sub, m0, GU_ROWS / 16, xs, xlen + XPAD, (kb_start + q) * GU_ROWS,
                 two);
        release(S, j);
      }
    }
    if constexpr (MODE != MODE_FP4) {
      const int cb = (warp >> 1) * 64 + m0;
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          if (h2 == 1 && !two) break;
#pragma unroll
          for (int r = 0; r < 4; ++r)
            out[(8 * h2 + 2 * tig + (r & 1)) * 256 + cb + 16 * m + g + ((r >> 1) << 3)] = d[m][h2][r];
        }
    }
  } else {
    // warp w: box w >> 2 (chunk 2c or 2c+1), columns [16*(w&3), +16), all 128 rows
    float d[2][4] = {};
    const uint32_t sub = uint32_t((warp >> 2) * (BLK_BYTES / 2));
    const int m0 = (warp & 3) * 16;
    if constexpr (MODE == MODE_FP4) {
      // NVFP4 block: 512 k of the warp's 16 down columns, A fragments from the codes
      for (int q = 0; q < nblk; ++q, ++j) {
        wait_full(S, j);
        const uint8_t* codes = stage_ptr(S, j);
        const uint8_t* scl = S.sm + fp4_scl_offset() + ((S.ring + j) % NSTAGE) * FP4_SCALE_BYTES;
        fp4_down_block(d, codes, scl, xs, xlen + XPAD, (kb_start + q) * FP4_DN_ROWS - kw);
        release(S, j);
      }
    } else {
      for (int q = 0; q < nblk; ++q, ++j) {
        const int kr = (kb_start + q) * DN_ROWS;  // first K row of this block
        if (MODE == MODE_DENSE && kr - kw >= xlen) {  // past the staged window (dense layers only; all warps)
          csync();  // every warp is done with the window
          kw = kr;
          xlen = min(ID - kw, H);
          stage_inputs<MODE>(S, it, xlen, kw);
        }
        wait_full(S, j);
        mma_tile(d, smem_u32(stage_ptr(S, j)) + sub, m0, 0, DN_ROWS / 16, xs, xlen + XPAD, kr - kw, two);
        release(S, j);
      }
    }
    const int cb = (warp >> 2) * 64 + m0;
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
      if (h2 == 1 && !two) break;
#pragma unroll
      for (int r = 0; r < 4; ++r) out[(8 * h2 + 2 * tig + (r & 1)) * 128 + cb + g + ((r >> 1) << 3)] = d[h2][r];
    }
  }
  csync();
  bool done = true;  // this CTA writes the item's outputs
  if (kb_start != 0 || nblk != it.KB) {
    // a piece of a split item: it opens this CTA's range (slot 0) or closes it (slot 1)
    float* P = partial_slot(S, blockIdx.x, j0 == 0 ? 0 : 1);
    for (int q = threadIdx.x; q < it.nt * ncol; q += NCONS) P[q] = out[q];
    done = ticket_add(item_ticket(p, it), uint32_t(nblk), uint32_t(it.KB), S.misc + 10);
    if (done) {
      // last arriver: add the item's pieces in block order
      if (threadIdx.x == 0) S.misc[11] = item_slots(S.L.n_total, S.nctas, S.b0 + j0 - kb_start, it.KB, S.plist);
      csync();
      const int npc = S.misc[11];
      for (int q = threadIdx.x; q < it.nt * ncol; q += NCONS) {
        float s = 0.f;
        for (int k0 = 0; k0 < npc; k0 += 8) {  // eight loads in flight, added in slot order
          float v[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) v[u] = k0 + u < npc ? __ldcg(S.pbank + (size_t)S.plist[k0 + u] * PSLOT + q) : 0.f;
#pragma unroll
          for (int u = 0; u < 8; ++u)
            if (k0 + u < npc) s += v[u];
        }
        out[q] = s;
      }
      csync();
    }
  }
  if (done) item_epilogue<MODE>(S, it, out);
  csync();
  // gate/up outputs of a token group complete: its down items may stage them (signalled per run)
  if (done && gu && S.dataflow) pend_done(S, gctr);
  // down outputs: the last item of a 128-column block combines that block for every token
  if (done && S.comb_items && !gu && ticket_last(p.tk_comb + it.c, uint32_t(S.comb_items), S.misc + 14, false)) {
    combine_block(p, S.inv, it.c);
    csync();
  }
}

// Consumers: work through this CTA's range of the step.
template <int MODE>
__device__ void consume(Stream& S) {
  int j = 0;
  while (j < S.nb) {
    int kind, idx, kb;
    block_kind(S.L, S.b0 + j, kind, idx, kb);
    const Item it = decode_item<MODE>(*S.p, S.meta, kind, idx);  // shared-memory lookups only
    if (kind == KIND_RT)
      run_router_block<MODE>(S, it, j);
    else
      run_segment<MODE>(S, it, kb, min(it.KB - kb, S.nb - j), j);
  }
  if (S.dataflow) flush_done(S);  // the step's last run of gate/up items
}

// Make L the current step: this CTA's range of its blocks.
__device__ __forceinline__ void set_step(Stream& S, const BlockList& L) {
  S.L = L;
  S.x_cls = -1;  // the staging buffer was reused between steps
  S.x_k0 = 0;
  S.b0 = range_begin(L.n_total, S.nctas, blockIdx.x);
  S.nb = range_begin(L.n_total, S.nctas, blockIdx.x + 1) - S.b0;
}

// Run the current step for the whole CTA: the producer lane streams (its first `pre` blocks
// were issued already), the consumers compute.
template <int MODE>
__device__ void run_step(Stream& S) {
  if (threadIdx.x >= NCONS) {
    if (threadIdx.x == NCONS) produce<MODE>(S, 0, S.nb);
  } else {
    consume<MODE>(S);
  }
  S.ring += S.nb;
  __syncthreads();
}

// Spread a bulk L2 prefetch of `bytes` (multiple of 16, below 2^32) at `base` over the grid
// (one thread; 32-bit arithmetic: a 64-bit division costs the producer warp microseconds).
__device__ __forceinline__ void prefetch_share(const void* base, uint32_t bytes) {
  const uint32_t per = ((bytes / gridDim.x) + 15u) & ~15u;
  const uint32_t a = per * blockIdx.x;
  if (a >= bytes) return;
  uint32_t n = per < bytes - a ? per : bytes - a;
  const uint8_t* src = static_cast<const uint8_t*>(base) + a;
  while (n) {
    const uint32_t c = n > 65536u ? 65536u : n;
    prefetch_l2_bulk(src, c);
    src += c;
    n -= c;
  }
}

// ---------------------------------------------------------------- routing
// Router logits (+ bias) of up to 4 tokens (list `toks`, count nt) into scores[t][e], then
// the top-K of each (warp t).  The sigmoid is strictly increasing, so ranking the fp32 logits
// gives the score order without the fp32 score saturating near 1; only the K chosen logits go
// through the sigmoid.  key = (order-preserving bits of the logit, 255 - expert): max =
// highest logit, lowest index on ties (-0 is folded into +0 so that they tie).
// All threads of the CTA call it.
// bias: the layer's router bias (or null); out_idx / out_w: the caller's copies of the routing
// (or null).
__device__ void route_tokens(const Params& p, const float* bias, int32_t* out_idx, float* out_w, uint8_t* sm,
                             const int* toks, int nt, int* s_idx, float* s_gw, bool write_global) {
  float* scores = reinterpret_cast<float*>(sm + Smem::scores);
  const int e = threadIdx.x;
  if (e < E) {
    for (int t = 0; t < nt; ++t) {
      const int tok = toks[t];
      float part[RT_NB];
#pragma unroll
      for (int rb = 0; rb < RT_NB; ++rb) part[rb] = __ldcg(p.RP + ((size_t)rb * STREAM_MAX_T + tok) * E + e);
      float l = 0.f;
#pragma unroll
      for (int rb = 0; rb < RT_NB; ++rb) l += part[rb];
      if (bias) l += bias[e];
      if (l == 0.f) l = 0.f;
      scores[t * E + e] = l;
    }
  }
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (warp < nt) {
    const int tok = toks[warp];
    // lane holds experts lane + 32 q; key = the logit's bits in an order-preserving unsigned form
    // (a non-NaN logit keys above 0, so 0 marks a taken expert).  Each round: the warp's largest
    // key (redux max over the lanes' own maxima), then the lowest expert holding it (redux min):
    // the order (logit desc, index asc), i.e. (score desc, index asc).
    uint32_t key[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const uint32_t u = __float_as_uint(scores[warp * E + lane + 32 * q]);
      key[q] = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    }
    uint32_t own = 0;  // this lane's largest remaining key
#pragma unroll
    for (int q = 0; q < 8; ++q) own = key[q] > own ? key[q] : own;
    float sel_s[K];
    int sel_e[K];
#pragma unroll
    for (int jj = 0; jj < K; ++jj) {
      const uint32_t best = __reduce_max_sync(0xffffffffu, own);
      uint32_t mine = 0xffffffffu;  // this lane's lowest expert with the best key
#pragma unroll
      for (int q = 7; q >= 0; --q)
        if (key[q] == best) mine = uint32_t(lane + 32 * q);
      const int ex = int(__reduce_min_sync(0xffffffffu, mine));
      sel_e[jj] = ex;
      sel_s[jj] = 1.0f / (1.0f + expf(-scores[warp * E + ex]));
      if ((ex & 31) == lane) {
        key[ex >> 5] = 0u;
        own = 0;
#pragma unroll
        for (int q = 0; q < 8; ++q) own = key[q] > own ? key[q] : own;
      }
    }
    if (lane == 0) {
      float sum = 0.f;
#pragma unroll
      for (int jj = 0; jj < K; ++jj) sum += sel_s[jj];
#pragma unroll
      for (int jj = 0; jj < K; ++jj) {
        const float g = sel_s[jj] / sum;
        if (s_idx) {
          s_idx[tok * K + jj] = sel_e[jj];
          s_gw[tok * K + jj] = g;
        }
        if (write_global) {
          p.topk_idx[tok * K + jj] = sel_e[jj];
          p.topk_w[tok * K + jj] = g;
          if (out_idx) out_idx[tok * K + jj] = sel_e[jj];
          if (out_w) out_w[tok * K + jj] = g;
        }
      }
    }
  }
  __syncthreads();
}

// Stable counting sort of the T*K (token, slot) pairs (expert ids in s_idx) by expert, in
// this CTA's shared memory: routing tables (Meta), perm (sorted row -> pair), inv.
// CTA 0 also publishes counts and offsets.  All threads of the CTA call it.
__device__ Meta build_tables(const Params& p, uint8_t* sm, uint16_t* perm, uint16_t* inv) {
  int* s_idx = reinterpret_cast<int*>(sm + Smem::s_idx);
  int* s_cnt = reinterpret_cast<int*>(sm + Smem::s_cnt);
  int* s_fill = reinterpret_cast<int*>(sm + Smem::s_fill);
  int* s_wcnt = reinterpret_cast<int*>(sm + Smem::s_wcnt);
  int* s_wsum = reinterpret_cast<int*>(sm + Smem::s_wsum);
  int* mbase = reinterpret_cast<int*>(sm + Smem::meta);
  int* me = mbase;
  int* moff = mbase + (E + 1);
  int* mcnt = mbase + 2 * (E + 1);
  int* mtgp = mbase + 3 * (E + 1);
  const int n = p.T * K;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool act = tid < E;  // thread == expert; the producer warp only synchronises
  if (act) s_cnt[tid] = 0;
  __syncthreads();
  if (act)
    for (int q = tid; q < n; q += E) {
      const int e = s_idx[q];
      if (e < 0 || e >= E) {
        record_status(p.status, ST_BOUNDS);
        continue;
      }
      atomicAdd(&s_cnt[e], 1);
    }
  __syncthreads();
  // exclusive scans over experts: counts, touched flags, token groups
  int c = 0, f = 0, ng = 0, ic = 0, jf = 0, kg = 0;
  if (act) {
    c = s_cnt[tid];
    f = c > 0 ? 1 : 0;
    ng = (c + group_rows(p.T) - 1) / group_rows(p.T);
    ic = c;
    jf = f;
    kg = ng;
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
  }
  __syncthreads();
  if (act) {
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
    if (f) {
      me[pos] = tid;
      moff[pos] = off_e;
      mcnt[pos] = c;
      mtgp[pos] = gpre;
    }
    if (tid == E - 1) {
      s_wsum[3 * NWARPS] = pos + f;
      s_wsum[3 * NWARPS + 1] = gpre + ng;
      mtgp[pos + f] = gpre + ng;
    }
    if (blockIdx.x == 0) {
      p.counts[tid] = c;
      p.offsets[tid] = off_e;
      if (p.out_counts) p.out_counts[tid] = c;
      if (tid == E - 1) p.offsets[E] = off_e + c;
    }
  }
  __syncthreads();
  // stable scatter, 256 pairs at a time in (t, j) order
  for (int base = 0; base < n; base += E) {
    if (act)
      for (int q = tid; q < NWARPS * E; q += E) s_wcnt[q] = 0;
    __syncthreads();
    const int pi = base + tid;
    int e = (act && pi < n) ? s_idx[pi] : -1;
    if (e >= E) e = -1;
    int r = 0;
    if (act) {
      const unsigned peers = __match_any_sync(0xffffffffu, e);
      r = __popc(peers & ((1u << lane) - 1u));
      if (e >= 0 && r == 0) s_wcnt[warp * E + e] = __popc(peers);
    }
    __syncthreads();
    if (e >= 0) {
      int before = 0;
      for (int w = 0; w < warp; ++w) before += s_wcnt[w * E + e];
      const int row = s_fill[e] + before + r;
      perm[row] = uint16_t(pi);
      inv[pi] = uint16_t(row);
    }
    __syncthreads();
    if (act) {
      int add = 0;
      for (int w = 0; w < NWARPS; ++w) add += s_wcnt[w * E + tid];
      s_fill[tid] += add;
    }
    __syncthreads();
  }
  Meta m;
  m.e = me;
  m.off = moff;
  m.cnt = mcnt;
  m.tgp = mtgp;
  m.U = s_wsum[3 * NWARPS];
  m.groups = s_wsum[3 * NWARPS + 1];
  __syncthreads();
  return m;
}

// A dense SwiGLU MLP layer (MODE_DENSE, width ID): the shared-expert steps alone -- step C
// the gate/up of the whole width, a barrier, step D the down projection, whose items write
// y = bf16(MLP(x') [+ x]) directly (no router, no routing, no combine).
template <int MODE>
__device__ void dense_layer(Stream& S, const Params& p, int ntg) {
  constexpr int sncb = ID / 128;
  S.dataflow = true;  // the down items wait for their token group's gate/up outputs: no barrier
  S.pbank = partial_bank(p, 0);
  {
    BlockList L;
    L.k_first = L.k_second = KIND_SGU;
    L.kb_first = L.kb_second = GU_KB;
    L.n_first = 0;
    L.n_total = ntg * sncb * GU_KB;
    S.first_slot = 12;
    trace_point(p, 6);
    set_step(S, L);
    run_step<MODE>(S);
  }
  trace_point(p, 7);
  {
    BlockList L;
    L.k_first = L.k_second = KIND_SD;
    L.kb_first = L.kb_second = ID / DN_ROWS;
    L.n_first = 0;
    L.n_total = ntg * OUT_NCB * (ID / DN_ROWS);
    set_step(S, L);
  }
  S.pbank = partial_bank(p, 1);
  trace_point(p, 8);
  S.first_slot = 13;
  run_step<MODE>(S);
  trace_point(p, 9);
  grid_done(p, S.misc + 13, 0, ntg);
  trace_point(p, 10);
}

// ================================================================ the fused decode kernel
// mode 0: the whole layer; mode 1: routing only (router, top-K, counts); a dense layer
// (MODE_DENSE) runs dense_layer instead.
template <int MODE>
__global__ void __launch_bounds__(NTHREADS, 1)
    decode_fused(const __grid_constant__ Params p, const __grid_constant__ StreamMaps maps, int mode) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = aligned_smem(smem_raw);
  Stream S;
  S.p = &p;
  S.maps = &maps;
  S.meta = Meta{};
  S.nctas = gridDim.x;
  S.ring = 0;
  S.first_slot = 11;
  S.sm = sm;
  S.full = reinterpret_cast<uint64_t*>(sm + Smem::full);
  S.empty = reinterpret_cast<uint64_t*>(sm + Smem::empty);
  S.misc = reinterpret_cast<int*>(sm + Smem::misc);
  S.plist = reinterpret_cast<int*>(sm + Smem::plist);
  S.out = reinterpret_cast<float*>(sm + out_offset(group_rows_mode(p.T, MODE)));
  S.comb_items = 0;
  S.dataflow = false;
  S.sig_ctr = nullptr;
  S.sig_n = 0;
  S.pbank = partial_bank(p, 0);
  uint16_t* perm = reinterpret_cast<uint16_t*>(sm + Smem::perm);
  uint16_t* inv = reinterpret_cast<uint16_t*>(sm + Smem::inv);
  float* gw = reinterpret_cast<float*>(sm + Smem::gw);
  int* s_idx = reinterpret_cast<int*>(sm + Smem::s_idx);
  S.perm = perm;
  S.inv = inv;
  S.gw = gw;
  const int T = p.T;
  const int ntg = (T + group_rows_mode(T, MODE) - 1) / group_rows_mode(T, MODE);
  const bool full = mode == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(S.full + s, 1);
      mbar_init(S.empty + s, NWARPS);
    }
    fence_mbar_init();
  }
  __syncthreads();
  trace_point(p, 0);
  pdl_wait();  // inputs of this forward and the workspace are ready
  trace_point(p, 1);
  if ((p.flags & FLAG_TEST_WAIT_TIMEOUT) && blockIdx.x == 0 && threadIdx.x == 0) test_wait_timeout(p.status);
  if constexpr (MODE == MODE_DENSE) {
    dense_layer<MODE>(S, p, ntg);
    return;
  }

  // ---- step A: router partial logits.  (The shared expert runs in steps C and D, beside the
  // routed experts: its blocks stream from L2 while the routed ones stream from HBM, and a
  // short step A starts the routing sooner; measured 908 vs 944 us over the decode sweep.)
  {
    if (full && threadIdx.x == NCONS + 1) {
      if (MODE == MODE_FP4)
        prefetch_share(p.q_sdown, uint32_t(IS) * H / 2);
      else
        prefetch_share(p.ws_down, uint32_t(IS) * H * 2);
    }
    BlockList L;
    L.k_first = L.k_second = KIND_RT;
    L.kb_first = L.kb_second = 1;
    L.n_first = L.n_total = ntg * RT_NB;
    set_step(S, L);
    run_step<MODE>(S);
  }
  trace_point(p, 2);
  if (!grid_sync(p, 1, S.misc + 12)) return;
  trace_point(p, 3);

  // ---- step B: routing, then this CTA's permutation tables
  int nbar = 1;
  if (T <= REDUNDANT_ROUTING_MAX_T) {
    int toks[REDUNDANT_ROUTING_MAX_T];
    for (int t = 0; t < T; ++t) toks[t] = t;
    route_tokens(p, p.router_bias, p.out_idx, p.out_w, sm, toks, T, s_idx, gw, blockIdx.x == 0);
  } else {
    int toks[4];
    int nt = 0;
    for (int t = blockIdx.x; t < T; t += gridDim.x) {
      toks[nt++] = t;
      if (nt == 4) {
        route_tokens(p, p.router_bias, p.out_idx, p.out_w, sm, toks, nt, nullptr, nullptr, true);
        nt = 0;
      }
    }
    if (nt) route_tokens(p, p.router_bias, p.out_idx, p.out_w, sm, toks, nt, nullptr, nullptr, true);
    if (!grid_sync(p, ++nbar, S.misc + 12)) return;
    for (int q = threadIdx.x; q < T * K; q += NTHREADS) {
      s_idx[q] = __ldcg(p.topk_idx + q);
      gw[q] = __ldcg(p.topk_w + q);
    }
    __syncthreads();
  }
  trace_point(p, 4);
  S.meta = build_tables(p, sm, perm, inv);
  trace_point(p, 5);
  if (!full) {
    grid_done(p, S.misc + 13);
    return;
  }

  // ---- step C: routed gate/up and the shared gate/up
  {
    BlockList L;
    const int kgu = kblocks_of<MODE>(p, KIND_GU);
    L.k_first = KIND_GU;
    L.kb_first = kgu;
    L.n_first = S.meta.groups * gu_ncb<MODE>() * kgu;
    L.k_second = KIND_SGU;
    L.kb_second = kgu;
    L.n_total = L.n_first + ntg * sgu_ncb<MODE>() * kgu;
    S.first_slot = 12;
    S.dataflow = true;  // gate/up items signal their token group; step D waits per group
    trace_point(p, 6);
    set_step(S, L);
    run_step<MODE>(S);
  }
  trace_point(p, 7);

  // ---- step D: routed down projection and the shared down projection, with no grid barrier
  // after step C: a CTA streams its down blocks (weights only) as soon as its step-C range is
  // done, and each down item waits only for the gate/up outputs of its own token group.  The
  // partial sums of split items use a second bank, since step-C pieces may still be being added.
  {
    BlockList L;
    const int kdn = kblocks_of<MODE>(p, KIND_DN), ksd = kblocks_of<MODE>(p, KIND_SD);
    L.k_first = KIND_DN;
    L.kb_first = kdn;
    L.n_first = S.meta.groups * OUT_NCB * kdn;
    L.k_second = KIND_SD;
    L.kb_second = ksd;
    L.n_total = L.n_first + ntg * OUT_NCB * ksd;
    set_step(S, L);
  }
  S.pbank = partial_bank(p, 1);
  trace_point(p, 8);
  // When the grid has a CTA for every down item, the combine of each 128-column block follows
  // its last down item (no further barrier); otherwise the whole grid combines after a barrier
  // (a ticket per item then costs each CTA a fence and an atomic per item: slower).
  S.comb_items = (S.meta.groups + ntg) * OUT_NCB <= S.nctas ? S.meta.groups + ntg : 0;
  S.first_slot = 13;
  run_step<MODE>(S);
  trace_point(p, 9);
  if (!S.comb_items) {
    if (!grid_sync(p, ++nbar, S.misc + 12)) return;
    trace_point(p, 14);
    combine_share(p, inv);
  }
  grid_done(p, S.misc + 13, S.meta.groups, ntg);
  trace_point(p, 10);
}

// ================================================================ the layer stack in one launch
// n_layers layers applied in place, x <- [x +] MoE_l([RMSNorm](x)), by one persistent cooperative
// kernel: each layer runs steps A-D as decode_fused does, and a grid barrier replaces the kernel
// boundary.  The combine gives each CTA whole token rows, so the same CTA normalises those rows
// for the next layer right away (no separate pre-norm pass).  Layer l's tensor maps, router bias
// and prefetch pointers come from a table in device memory; everything else is the launch's
// parameters (read from the constant bank: a shared-memory copy of them measured 3-4 % slower).

// The stack runs in one launch at every decode size.  Measured on B300 (12 layers, pre-norm +
// residual, us per layer, one launch against per-layer calls of decode_fused): T = 1 32.8 vs
// 38.5, T = 4 50.7 vs 60.3, T = 32 156.8 vs 160.5, T = 64 220.8 vs 224.8, T = 256 301.7 vs 303.8.

// Per-layer entry of the stack's device table (aligned as its tensor maps; the table starts on a
// 256-byte boundary).
struct LayerTab {
  StreamMaps maps;
  const float* router_bias;
  const bf16* w_router;
  const bf16* ws_gate;
  const bf16* ws_up;
  const bf16* ws_down;
};
static_assert(alignof(LayerTab) >= 64 && alignof(LayerTab) <= 256, "tensor maps stay aligned in the table");


// r = bf16(v / sqrt(mean(v^2) + eps)) of one token row whose eight values v (bf16, packed)
// column chunk threadIdx.x holds, written to xn: the reduction of rmsnorm_kernel (thread i sums
// its chunk in order, a butterfly over the warp, the eight warp sums in order).  Consumers only;
// `red` is [NWARPS] floats of shared scratch.
__device__ __forceinline__ void norm_row(const Params& p, int t, uint4 v, float* red) {
  float f[8];
  bf16x8_to_f32(v, f);
  float ss = 0.f;
#pragma unroll
  for (int q = 0; q < 8; ++q) ss = fmaf(f[q], f[q], ss);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  csync();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < NWARPS; ++w) tot += red[w];
  const float d = sqrtf(tot / float(H) + p.rms_eps);
  uint32_t packed[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const __nv_bfloat162 b = __floats2bfloat162_rn(f[2 * q] / d, f[2 * q + 1] / d);
    packed[q] = *reinterpret_cast<const uint32_t*>(&b);
  }
  *(reinterpret_cast<uint4*>(p.xn + (size_t)t * H) + threadIdx.x) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
  csync();  // red is reused by the next row
}

__global__ void __launch_bounds__(NTHREADS, 1)
    decode_stack(const __grid_constant__ Params base, const LayerTab* __restrict__ tab, int n_layers) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = aligned_smem(smem_raw);
  const int T = base.T;
  const int G = group_rows(T);
  const int ntg = (T + G - 1) / G;
  const bool prenorm = (base.flags & 1u) != 0;  // FLINT_MOE_FLAG_PRE_RMSNORM
  const Params& p = base;
  Stream S;
  S.p = &base;
  S.meta = Meta{};
  S.nctas = gridDim.x;
  S.ring = 0;
  S.first_slot = 11;
  S.sm = sm;
  S.full = reinterpret_cast<uint64_t*>(sm + Smem::full);
  S.empty = reinterpret_cast<uint64_t*>(sm + Smem::empty);
  S.misc = reinterpret_cast<int*>(sm + Smem::misc);
  S.plist = reinterpret_cast<int*>(sm + Smem::plist);
  S.out = reinterpret_cast<float*>(sm + out_offset(G));
  S.dataflow = false;
  S.sig_ctr = nullptr;
  S.sig_n = 0;
  S.pbank = partial_bank(base, 0);
  S.comb_items = 0;  // the combine always follows a barrier here: it also normalises
  uint16_t* perm = reinterpret_cast<uint16_t*>(sm + Smem::perm);
  uint16_t* inv = reinterpret_cast<uint16_t*>(sm + Smem::inv);
  float* gw = reinterpret_cast<float*>(sm + Smem::gw);
  int* s_idx = reinterpret_cast<int*>(sm + Smem::s_idx);
  S.perm = perm;
  S.inv = inv;
  S.gw = gw;
  if (threadIdx.x == 0) {
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(S.full + s, 1);
      mbar_init(S.empty + s, NWARPS);
    }
    fence_mbar_init();
  }
  __syncthreads();
  trace_point(p, 0);
  pdl_wait();
  trace_point(p, 1);
  if ((base.flags & FLAG_TEST_WAIT_TIMEOUT) && blockIdx.x == 0 && threadIdx.x == 0) test_wait_timeout(base.status);
  int nbar = 0;
  // the first layer's pre-norm: whole rows per CTA
  if (prenorm) {
    if (threadIdx.x < NCONS)
      for (int t = blockIdx.x; t < T; t += gridDim.x)
        norm_row(p, t, __ldcg(reinterpret_cast<const uint4*>(p.x + (size_t)t * H) + threadIdx.x), S.out);
    if (!grid_sync(p, ++nbar, S.misc + 12)) return;
  }
  for (int l = 0; l < n_layers; ++l) {
    const float* bias = tab[l].router_bias;
    int32_t* out_idx = base.out_idx ? base.out_idx + (size_t)l * T * K : nullptr;
    float* out_w = base.out_w ? base.out_w + (size_t)l * T * K : nullptr;
    S.maps = &tab[l].maps;
    if (threadIdx.x == NCONS) {  // the layer's descriptors are read from device memory by every TMA issue
      prefetch_tensormap(&S.maps->wr);
      prefetch_tensormap(&S.maps->wg);
      prefetch_tensormap(&S.maps->wu);
      prefetch_tensormap(&S.maps->wd);
      prefetch_tensormap(&S.maps->wsg);
      prefetch_tensormap(&S.maps->wsu);
      prefetch_tensormap(&S.maps->wsd);
    }
    // ---- step A: router partial logits
    {
      if (l == 0 && threadIdx.x == NCONS + 1) prefetch_share(tab[l].ws_down, uint32_t(IS) * H * 2);
      BlockList L;
      L.k_first = L.k_second = KIND_RT;
      L.kb_first = L.kb_second = 1;
      L.n_first = L.n_total = ntg * RT_NB;
      S.first_slot = 11;
      set_step(S, L);
      run_step<MODE_MOE>(S);
    }
    trace_point(p, 2);
    if (!grid_sync(p, ++nbar, S.misc + 12)) return;
    trace_point(p, 3);
    // ---- step B: routing, then this CTA's permutation tables
    if (T <= REDUNDANT_ROUTING_MAX_T) {
      int toks[REDUNDANT_ROUTING_MAX_T];
      for (int t = 0; t < T; ++t) toks[t] = t;
      route_tokens(p, bias, out_idx, out_w, sm, toks, T, s_idx, gw, blockIdx.x == 0);
    } else {
      int toks[4];
      int nt = 0;
      for (int t = blockIdx.x; t < T; t += gridDim.x) {
        toks[nt++] = t;
        if (nt == 4) {
          route_tokens(p, bias, out_idx, out_w, sm, toks, nt, nullptr, nullptr, true);
          nt = 0;
        }
      }
      if (nt) route_tokens(p, bias, out_idx, out_w, sm, toks, nt, nullptr, nullptr, true);
      if (!grid_sync(p, ++nbar, S.misc + 12)) return;
      for (int q = threadIdx.x; q < T * K; q += NTHREADS) {
        s_idx[q] = __ldcg(p.topk_idx + q);
        gw[q] = __ldcg(p.topk_w + q);
      }
      __syncthreads();
    }
    trace_point(p, 4);
    S.meta = build_tables(p, sm, perm, inv);
    trace_point(p, 5);
    // ---- step C: routed gate/up and the shared gate/up
    {
      BlockList L;
      L.k_first = KIND_GU;
      L.kb_first = GU_KB;
      L.n_first = S.meta.groups * GU_NCB * GU_KB;
      L.k_second = KIND_SGU;
      L.kb_second = GU_KB;
      L.n_total = L.n_first + ntg * SGU_NCB * GU_KB;
      S.first_slot = 12;
      S.pbank = partial_bank(base, 0);
      S.dataflow = true;  // gate/up items signal their token group; step D waits per group
      trace_point(p, 6);
      set_step(S, L);
      run_step<MODE_MOE>(S);
    }
    trace_point(p, 7);
    // ---- step D, with no grid barrier after step C (the dataflow of decode_fused)
    {
      BlockList L;
      L.k_first = KIND_DN;
      L.kb_first = DN_KB;
      L.n_first = S.meta.groups * OUT_NCB * DN_KB;
      L.k_second = KIND_SD;
      L.kb_second = SD_KB;
      L.n_total = L.n_first + ntg * OUT_NCB * SD_KB;
      set_step(S, L);
    }
    S.pbank = partial_bank(base, 1);
    trace_point(p, 8);
    S.first_slot = 13;
    run_step<MODE_MOE>(S);
    S.dataflow = false;
    trace_point(p, 9);
    // The next layer's router and shared-expert weights (13 MB) do not depend on this layer's
    // results: a CTA that has finished its step-D range asks L2 for its share of them, while HBM
    // serves the other CTAs' last down blocks, so that the next layer's router step and shared
    // blocks read from L2.
    if (l + 1 < n_layers && threadIdx.x == NCONS + 1) {
      const LayerTab& nx = tab[l + 1];
      prefetch_share(nx.w_router, uint32_t(H) * E * 2);
      prefetch_share(nx.ws_gate, uint32_t(H) * IS * 2);
      prefetch_share(nx.ws_up, uint32_t(H) * IS * 2);
      prefetch_share(nx.ws_down, uint32_t(IS) * H * 2);
    }
    if (!grid_sync(p, ++nbar, S.misc + 12)) return;
    trace_point(p, 14);
    // every step-D wait of this layer is over: clear the token-group counters for the next layer
    // (the barrier at the end of the combine orders these stores before its first signal)
    for (int i = blockIdx.x * NTHREADS + threadIdx.x; i < S.meta.groups; i += gridDim.x * NTHREADS) p.hdone[i] = 0u;
    for (int i = blockIdx.x * NTHREADS + threadIdx.x; i < ntg; i += gridDim.x * NTHREADS) p.hsdone[i] = 0u;
    // ---- the combine by whole rows, and the next layer's pre-norm of the same rows
    const bool norm_next = prenorm && l + 1 < n_layers;
    if (threadIdx.x < NCONS)
      for (int t = blockIdx.x; t < T; t += gridDim.x) {
        const uint4 v = combine8(p, inv, t, threadIdx.x * 8);
        if (norm_next) norm_row(p, t, v, S.out);
      }
    if (l + 1 < n_layers && !grid_sync(p, ++nbar, S.misc + 12)) return;
  }
  grid_done(p, S.misc + 13);
  trace_point(p, 10);
}

// ================================================================ RMSNorm (pre-norm layers)
// xn[t] = bf16(x[t] / sqrt(mean(x[t]^2) + eps)), unit weight; one CTA of 256 threads per token.
__global__ void __launch_bounds__(256) rmsnorm_kernel(const __grid_constant__ Params p) {
  __shared__ float s_w[8];
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
  for (int w = 0; w < 8; ++w) tot += s_w[w];
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
