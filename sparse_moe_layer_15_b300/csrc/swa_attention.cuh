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
// loads each, many resident per SM.  A CTA stages its chunk's K and V rows (256 bytes each,
// 16-byte loads, rows padded to spread shared-memory banks) and the group's 8 query rows; warp
// w is query head 8g + w: each lane scores one or two slots (a 128-long dot product), the warp
// takes the chunk's max and sum of e^(s - max), and each lane accumulates 4 output dimensions
// over the chunk's slots.  The chunk's unnormalised output, max and sum go to the workspace; an
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
constexpr int NT = GQ * 32;                 // 256 threads: one warp per query head of the group
constexpr int ROWB = HD * 2 + 16;           // padded shared-memory row (bytes)
constexpr int PSTRIDE = HD + 4;             // floats of one chunk's partial: o[128], m, l, pad
static_assert(NSPLIT * CH == W, "the chunks tile the window");
static_assert(CH <= 64, "at most two slots per lane");

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

__device__ __forceinline__ float dot8(uint4 a, uint4 b, float acc) {
  float fa[8], fb[8];
  bf16x8_to_f32(a, fa);
  bf16x8_to_f32(b, fb);
#pragma unroll
  for (int i = 0; i < 8; ++i) acc = fmaf(fa[i], fb[i], acc);
  return acc;
}

__global__ void __launch_bounds__(NT) decode_kernel(const __grid_constant__ Params p) {
  __shared__ __align__(16) uint8_t ks[CH * ROWB];
  __shared__ __align__(16) uint8_t vs[CH * ROWB];
  __shared__ __align__(16) uint4 qs[GQ * HD / 8];
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

  // ---- stage K and V rows of the chunk's valid slots, and the group's query rows
  constexpr int RV = HD / 8;  // 16-byte pieces per row
  {
    const uint4* kg = reinterpret_cast<const uint4*>(p.k + ((size_t)b * W + j0) * NKV * HD + (size_t)g * HD);
    const uint4* vg = reinterpret_cast<const uint4*>(p.v + ((size_t)b * W + j0) * NKV * HD + (size_t)g * HD);
    constexpr int PER = (2 * CH * RV + NT - 1) / NT;
    uint4 buf[PER];
#pragma unroll
    for (int u = 0; u < PER; ++u) {  // all loads in flight before the stores
      const int i = tid + u * NT;
      const int r = i / RV, c = i % RV;
      const int j = r < CH ? r : r - CH;
      buf[u] = make_uint4(0, 0, 0, 0);
      if (i < 2 * CH * RV && j < nk) buf[u] = __ldcs((r < CH ? kg : vg) + (size_t)j * NKV * RV + c);
    }
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      const int i = tid + u * NT;
      if (i >= 2 * CH * RV) break;
      const int r = i / RV, c = i % RV;
      const int j = r < CH ? r : r - CH;
      *reinterpret_cast<uint4*>((r < CH ? ks : vs) + j * ROWB + c * 16) = buf[u];
    }
    if (tid < GQ * RV)
      qs[tid] = __ldg(reinterpret_cast<const uint4*>(p.q + ((size_t)b * NH + (size_t)g * GQ) * HD) + tid);
  }
  __syncthreads();

  // ---- warp w: query head h = 8g + w; lane: slots lane and lane + 32
  const int h = g * GQ + warp;
  const uint4* qrow = qs + warp * RV;
  float s[2];
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int j = lane + 32 * t;
    s[t] = -INFINITY;
    if (j < nk) {
      const uint4* krow = reinterpret_cast<const uint4*>(ks + j * ROWB);
      float acc = 0.f;
#pragma unroll
      for (int c = 0; c < RV; ++c) acc = dot8(qrow[c], krow[c], acc);
      s[t] = acc * SCALE;
    }
  }
  float m = fmaxf(s[0], s[1]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  float e[2];
#pragma unroll
  for (int t = 0; t < 2; ++t) e[t] = (lane + 32 * t < nk) ? expf(s[t] - m) : 0.f;
  float l = e[0] + e[1];
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
  // o[4 lane .. 4 lane + 3] = sum_j e_j v_j, slots in order
  float o[4] = {0.f, 0.f, 0.f, 0.f};
  for (int j = 0; j < nk; ++j) {
    const float ej = __shfl_sync(0xffffffffu, j < 32 ? e[0] : e[1], j & 31);
    const uint2 vv = *reinterpret_cast<const uint2*>(vs + j * ROWB + lane * 8);
    o[0] = fmaf(ej, __uint_as_float(vv.x << 16), o[0]);
    o[1] = fmaf(ej, __uint_as_float(vv.x & 0xFFFF0000u), o[1]);
    o[2] = fmaf(ej, __uint_as_float(vv.y << 16), o[2]);
    o[3] = fmaf(ej, __uint_as_float(vv.y & 0xFFFF0000u), o[3]);
  }
  float* pp = p.part + (((size_t)b * NH + h) * NSPLIT + split) * PSTRIDE;
  *reinterpret_cast<float4*>(pp + 4 * lane) = make_float4(o[0], o[1], o[2], o[3]);
  if (lane == 0) {
    pp[HD] = m;  // -inf for a chunk without valid slots (then l = 0 and o = 0)
    pp[HD + 1] = l;
  }

  // ---- the last of the NSPLIT CTAs of (b, g) merges the chunks with the sink
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
  const float sink = __ldg(p.sinks + h);
  const float* ph = p.part + ((size_t)b * NH + h) * NSPLIT * PSTRIDE;
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
    const float w = ms[c] == -INFINITY ? 0.f : expf(ms[c] - M);
    const float4 oc = __ldcg(reinterpret_cast<const float4*>(ph + c * PSTRIDE + 4 * lane));
    L = fmaf(w, __ldcg(ph + c * PSTRIDE + HD + 1), L);
    O[0] = fmaf(w, oc.x, O[0]);
    O[1] = fmaf(w, oc.y, O[1]);
    O[2] = fmaf(w, oc.z, O[2]);
    O[3] = fmaf(w, oc.w, O[3]);
  }
  const float inv = 1.0f / L;
  const __nv_bfloat162 r0 = __floats2bfloat162_rn(O[0] * inv, O[1] * inv);
  const __nv_bfloat162 r1 = __floats2bfloat162_rn(O[2] * inv, O[3] * inv);
  uint2 packed;
  packed.x = *reinterpret_cast<const uint32_t*>(&r0);
  packed.y = *reinterpret_cast<const uint32_t*>(&r1);
  *reinterpret_cast<uint2*>(p.out + ((size_t)b * NH + h) * HD + 4 * lane) = packed;
}

}  // namespace swa
}  // namespace flint
