// Decode attention of the sliding-window layers (serving-kit post, "The architecture, from the
// config": 35 of the 49 layers attend to a 513-token window, the current token plus 512 back;
// 32 query heads share 4 KV heads of dimension 128; learned per-head attention sinks.  News
// article "Recursive opens Flint, a 40B coding model with 2.5B active", section "What runs on
// each token": a sink is a slot that can take attention no real token needs).
//
// One decode step of B sequences: for every sequence b and query head h (KV head g = h / 8),
//   out[b][h] = sum_j e^(s_j - m) v_j / (e^(sink_h - m) + sum_j e^(s_j - m)),
//   s_j = q[b][h] . k_j / sqrt(128),  m = max(sink_h, max_j s_j),
// over the valid slots j of the sequence's ring cache (position p in slot p mod 513; the slots
// 0 .. min(pos[b] + 1, 513) - 1 are valid).  The sink is a logit of the softmax denominator with
// no value.  q and k arrive normalised and rotated (the per-head QK RMSNorm and RoPE belong to
// the projections).
//
// The step reads 513 x 4 x 128 x 2 x 2 = 525 KB of cache per full sequence and does about 8
// MFLOP: HBM-bound.  Work split: one CTA per (57-slot chunk, KV head, sequence) -- 9 chunks
// cover the 513 slots exactly -- so a batch of B sequences launches 36 B CTAs of 29 KB of
// loads each, several resident per SM.  A CTA stages its chunk's K and V rows (256 bytes each,
// 16-byte loads, rows padded to spread shared-memory banks) and the group's 8 query rows, then
// runs both contractions as bf16 warp MMAs (m16n8k16, fp32 accumulate) with the 8 heads as the
// rows of a 16-row tile: S = Q K^T split over the warps by slots, the chunk's softmax statistics
// reduced across the warps in fp32, the probabilities rounded to bf16, O = P V split over the
// warps by output dimensions.  The chunk's unnormalised output, max and sum go to the workspace; an
// integer ticket per (sequence, KV head) elects the last of the 9 CTAs, which merges the chunks
// in chunk order together with the sink: deterministic, no floating-point atomics.
#pragma once

#include "common.cuh"

namespace flint {
namespace swa {

constexpr int NH = 32;
constexpr int NKV = 4;
constexpr int HD = 128;
constexpr int W = 513;
constexpr int GQ = NH / NKV;                // 8 query heads per KV head
constexpr int CH = 57;                      // cached slots per CTA
constexpr int NSPLIT = (W + CH - 1) / CH;   // 9 chunks, 9 x 57 = 513
constexpr int NT = GQ * 32;                 // 256 threads (8 warps)
constexpr int PSTRIDE = HD + 4;             // floats of one chunk's partial: o[128], m, l, pad
static_assert(NSPLIT * CH == W, "the chunks tile the window");
static_assert(CH <= 64, "a chunk fits the 64-slot MMA tiles");

struct Params {
  const bf16* q;        // [B][NH][HD]
  const bf16* k;        // [B][W][NKV][HD]
  const bf16* v;        // [B][W][NKV][HD]
  const float* sinks;   // [NH]
  const int32_t* pos;   // [B]
  bf16* out;            // [B][NH][HD]
  int B;
  float* part;          // [B][NH][NSPLIT][PSTRIDE] chunk partials
  uint32_t* ticket;     // [B][NKV], zero between calls (the last arriver resets)
  uint32_t* status;     // device status word
};

// 1 / sqrt(128)
constexpr float SCALE = 0.08838834764831845f;
constexpr int KP = 64;       // slots of a chunk padded to the MMA tiles (slots >= 57 are zero)
constexpr int RS = HD + 8;   // bf16 row stride of the staged K, V and query rows (272 bytes: banks spread)
constexpr int PS = KP + 8;   // bf16 row stride of the probabilities

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// A fragment (16 x 16, row-major, row stride `rs` bf16) of rows 0..15, columns [k0, k0 + 16).
__device__ __forceinline__ void frag_a(uint32_t base, int rs, int k0, uint32_t (&a)[4]) {
  const int lane = threadIdx.x & 31, q = lane >> 3;
  ldsm_x4(base + uint32_t((((q & 1) * 8 + (lane & 7)) * rs + k0 + (q >> 1) * 8) * 2), a);
}

// The chunk's attention with the group's 8 query heads as the rows of 16-row MMA tiles (rows 8..15
// zero): S = Q K^T over 128 dimensions (warp w: slots [8w, 8w + 8)), the chunk's softmax across
// the warps (fp32), P rounded to bf16, O = P V over the 64 padded slots (warp w: dimensions
// [16w, 16w + 16)).
__global__ void __launch_bounds__(NT) decode_kernel(const __grid_constant__ Params p) {
  __shared__ __align__(16) bf16 ks[KP * RS];
  __shared__ __align__(16) bf16 vs[KP * RS];
  __shared__ __align__(16) bf16 qs[16 * RS];
  __shared__ __align__(16) bf16 ps[16 * PS];
  __shared__ float red_m[GQ][8], red_l[GQ][8];
  __shared__ int s_last;
  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int pb = __ldg(p.pos + b);
  if (pb < 0) {
    if (tid == 0) record_status(p.status, ST_BOUNDS);
    pb = 0;
  }
  const int n = pb + 1 < W ? pb + 1 : W;
  const int j0 = split * CH;
  const int nk = n - j0 < 0 ? 0 : (n - j0 < CH ? n - j0 : CH);  // valid slots of this chunk

  // ---- stage K and V rows (zero beyond the valid slots), the group's 8 query rows (+ 8 zero rows),
  // and zero probability rows 8..15
  constexpr int RV = HD / 8;  // 16-byte pieces per row
  {
    const uint4* kg = reinterpret_cast<const uint4*>(p.k + ((size_t)b * W + j0) * NKV * HD + (size_t)g * HD);
    const uint4* vg = reinterpret_cast<const uint4*>(p.v + ((size_t)b * W + j0) * NKV * HD + (size_t)g * HD);
    constexpr int PER = (2 * KP * RV + NT - 1) / NT;  // 8
    uint4 buf[PER];
#pragma unroll
    for (int u = 0; u < PER; ++u) {  // all loads in flight before the stores
      const int i = tid + u * NT;
      const int r = i / RV, c = i % RV;
      const int j = r < KP ? r : r - KP;
      buf[u] = make_uint4(0, 0, 0, 0);
      if (j < nk) buf[u] = __ldcs((r < KP ? kg : vg) + (size_t)j * NKV * RV + c);
    }
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      const int i = tid + u * NT;
      const int r = i / RV, c = i % RV;
      const int j = r < KP ? r : r - KP;
      *reinterpret_cast<uint4*>((r < KP ? ks : vs) + j * RS + c * 8) = buf[u];
    }
    const uint4 zero = make_uint4(0, 0, 0, 0);
    {
      const int r = tid / RV, c = tid % RV;  // 256 threads: 16 rows x 16 pieces
      *reinterpret_cast<uint4*>(qs + r * RS + c * 8) =
          r < GQ ? __ldg(reinterpret_cast<const uint4*>(p.q + ((size_t)b * NH + (size_t)g * GQ + r) * HD) + c) : zero;
    }
    if (tid < 8 * (KP / 8)) *reinterpret_cast<uint4*>(ps + (8 + tid / (KP / 8)) * PS + (tid % (KP / 8)) * 8) = zero;
  }
  __syncthreads();

  // ---- S = Q K^T: warp w, slots [8w, 8w + 8)
  const int row = lane >> 2;          // query head within the group (C-fragment rows 0..7)
  const int cq = 2 * (lane & 3);      // C-fragment column pair
  float sacc[4] = {0.f, 0.f, 0.f, 0.f};
  {
    const uint32_t qb = smem_u32(qs), kb = smem_u32(ks);
    const int q = lane >> 3;
#pragma unroll
    for (int k0 = 0; k0 < HD; k0 += 32) {
      uint32_t a0[4], a1[4], bb[4];
      frag_a(qb, RS, k0, a0);
      frag_a(qb, RS, k0 + 16, a1);
      ldsm_x4(kb + uint32_t(((warp * 8 + (lane & 7)) * RS + k0 + q * 8) * 2), bb);
      mma16816(sacc, a0, bb[0], bb[1]);
      mma16816(sacc, a1, bb[2], bb[3]);
    }
  }
  const int jA = warp * 8 + cq;
  const float s0 = jA < nk ? sacc[0] * SCALE : -INFINITY;
  const float s1 = jA + 1 < nk ? sacc[1] * SCALE : -INFINITY;
  float mw = fmaxf(s0, s1);
  mw = fmaxf(mw, __shfl_xor_sync(0xffffffffu, mw, 1));
  mw = fmaxf(mw, __shfl_xor_sync(0xffffffffu, mw, 2));
  if ((lane & 3) == 0) red_m[warp][row] = mw;
  __syncthreads();
  float m = red_m[0][row];
#pragma unroll
  for (int w = 1; w < GQ; ++w) m = fmaxf(m, red_m[w][row]);
  // m = -inf only when the chunk has no valid slot: every probability is 0 then
  const float p0 = jA < nk ? expf(s0 - m) : 0.f;
  const float p1 = jA + 1 < nk ? expf(s1 - m) : 0.f;
  float lw = p0 + p1;
  lw += __shfl_xor_sync(0xffffffffu, lw, 1);
  lw += __shfl_xor_sync(0xffffffffu, lw, 2);
  if ((lane & 3) == 0) red_l[warp][row] = lw;
  *reinterpret_cast<__nv_bfloat162*>(ps + row * PS + jA) = __floats2bfloat162_rn(p0, p1);
  __syncthreads();

  // ---- O = P V: warp w, dimensions [16w, 16w + 16) (two 8-column tiles)
  float o[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
  {
    const uint32_t pb0 = smem_u32(ps), vb = smem_u32(vs);
    const int q = lane >> 3;
#pragma unroll
    for (int k0 = 0; k0 < KP; k0 += 32) {
      uint32_t a0[4], a1[4];
      frag_a(pb0, PS, k0, a0);
      frag_a(pb0, PS, k0 + 16, a1);
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        uint32_t bb[4];
        ldsm_x4_t(vb + uint32_t(((k0 + q * 8 + (lane & 7)) * RS + warp * 16 + t * 8) * 2), bb);
        mma16816(o[t], a0, bb[0], bb[1]);
        mma16816(o[t], a1, bb[2], bb[3]);
      }
    }
  }
  // chunk partials: o (unnormalised, fp32), m, l per query head
  const int h = g * GQ + row;
  float* pp = p.part + (((size_t)b * NH + h) * NSPLIT + split) * PSTRIDE;
#pragma unroll
  for (int t = 0; t < 2; ++t)
    *reinterpret_cast<float2*>(pp + warp * 16 + t * 8 + cq) = make_float2(o[t][0], o[t][1]);
  if (warp == 0 && (lane & 3) == 0) {
    float l = red_l[0][row];
#pragma unroll
    for (int w = 1; w < GQ; ++w) l += red_l[w][row];
    pp[HD] = m;  // -inf for a chunk without valid slots (then l = 0 and o = 0)
    pp[HD + 1] = l;
  }

  // ---- the last of the NSPLIT CTAs of (b, g) merges the chunks with the sink (warp w: head 8g + w,
  // lane: dimensions 4 lane .. 4 lane + 3), in chunk order
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    uint32_t* tk = p.ticket + (size_t)b * NKV + g;
    const uint32_t prev = atomicAdd(tk, 1u);
    s_last = prev == NSPLIT - 1;
    if (s_last) *tk = 0u;  // every CTA of (b, g) has arrived: ready for the next call
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const int hm = g * GQ + warp;
  const float sink = __ldg(p.sinks + hm);
  const float* ph = p.part + ((size_t)b * NH + hm) * NSPLIT * PSTRIDE;
  float ms[NSPLIT], M = sink;
#pragma unroll
  for (int c = 0; c < NSPLIT; ++c) {
    ms[c] = __ldcg(ph + c * PSTRIDE + HD);
    M = fmaxf(M, ms[c]);
  }
  float L = expf(sink - M);
  float O[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int c = 0; c < NSPLIT; ++c) {
    const float wgt = ms[c] == -INFINITY ? 0.f : expf(ms[c] - M);
    const float4 oc = __ldcg(reinterpret_cast<const float4*>(ph + c * PSTRIDE + 4 * lane));
    L = fmaf(wgt, __ldcg(ph + c * PSTRIDE + HD + 1), L);
    O[0] = fmaf(wgt, oc.x, O[0]);
    O[1] = fmaf(wgt, oc.y, O[1]);
    O[2] = fmaf(wgt, oc.z, O[2]);
    O[3] = fmaf(wgt, oc.w, O[3]);
  }
  const float inv = 1.0f / L;
  const __nv_bfloat162 r0 = __floats2bfloat162_rn(O[0] * inv, O[1] * inv);
  const __nv_bfloat162 r1 = __floats2bfloat162_rn(O[2] * inv, O[3] * inv);
  uint2 packed;
  packed.x = *reinterpret_cast<const uint32_t*>(&r0);
  packed.y = *reinterpret_cast<const uint32_t*>(&r1);
  *reinterpret_cast<uint2*>(p.out + ((size_t)b * NH + hm) * HD + 4 * lane) = packed;
}

}  // namespace swa
}  // namespace flint
