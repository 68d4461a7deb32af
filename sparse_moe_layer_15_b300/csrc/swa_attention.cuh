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
// MFLOP: HBM-bound.  The window is cut into 9 chunks of 57 slots.  A CTA takes one (sequence, KV
// head) and walks its chunks with a running softmax, loading chunk c + 1 (cp.async, 16 bytes per
// thread, rows padded to spread shared-memory banks) while chunk c is computed; both
// contractions are bf16 warp MMAs (m16n8k16, fp32 accumulate) with the 8 heads of the group as the
// rows of a 16-row tile: S = Q K^T split over the warps by slots, the chunk's row max reduced
// across the warps, P rounded to bf16, O = P V split over the warps by output dimensions.  When a
// batch has fewer (sequence, KV head) pairs than SMs, each pair is split over 9 CTAs of one chunk
// each: a CTA writes its unnormalised output, max and sum to the workspace, and an integer
// ticket per (sequence, KV head) elects the last of them, which merges the chunks in chunk order
// together with the sink.  Deterministic either way, no floating-point atomics.
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
static_assert((2 * KP * (HD / 8)) % NT == 0, "a chunk's copies are whole rounds of the CTA");

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

// Shared memory (dynamic): two chunk buffers of K and V rows, the query rows, the probabilities.
struct Smem {
  static constexpr int kv = 0;                              // [2 buffers][K | V][KP][RS] bf16
  static constexpr int qs = kv + 2 * 2 * KP * RS * 2;      // [16][RS] bf16
  static constexpr int ps = qs + 16 * RS * 2;              // [16][PS] bf16
  static constexpr int red = ps + 16 * PS * 2;             // [2][GQ][8] f32
  static constexpr int bytes = red + 2 * GQ * 8 * 4 + 16;
};
constexpr int SMEM_BYTES = Smem::bytes;

// One CTA per (split, KV head, sequence) walks chunks [split * cpc, +cpc) of the 9 (cpc = 9 /
// splits): chunk c + 1 is loaded (cp.async, slots beyond the valid ones zero-filled) while chunk
// c is computed.  Per chunk, with the group's 8 query heads as the rows of 16-row MMA tiles (rows
// 8..15 zero): S = Q K^T (warp w: slots [8w, 8w + 8)), the chunk's row max across the warps, the
// running softmax (max m, sum l, output O rescaled by e^(m_old - m_new)), P rounded to bf16, O +=
// P V (warp w: dimensions [16w, 16w + 16)).  One split: the CTA writes the output with the sink;
// several: its (O, m, l) go to the workspace and the last CTA of (b, g) merges them.
__global__ void __launch_bounds__(NT) decode_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(16) uint8_t smem[];
  bf16* kvb = reinterpret_cast<bf16*>(smem + Smem::kv);
  bf16* qs = reinterpret_cast<bf16*>(smem + Smem::qs);
  bf16* ps = reinterpret_cast<bf16*>(smem + Smem::ps);
  float* red = reinterpret_cast<float*>(smem + Smem::red);  // [0]: row maxima, [1]: row sums
  __shared__ int s_last;
  const int nsplit = gridDim.x, split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int cpc = NSPLIT / nsplit;  // chunks per CTA
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int pb = __ldg(p.pos + b);
  if (pb < 0) {
    if (tid == 0) record_status(p.status, ST_BOUNDS);
    pb = 0;
  }
  const int n = pb + 1 < W ? pb + 1 : W;
  constexpr int RV = HD / 8;  // 16-byte pieces per row

  // chunk c -> buffer c & 1 (K rows, then V rows; slots beyond the valid ones zero-filled)
  auto load_chunk = [&](int c) {
    const int j0 = c * CH;
    const int nk = n - j0 < 0 ? 0 : (n - j0 < CH ? n - j0 : CH);
    const bf16* kg = p.k + ((size_t)b * W + j0) * NKV * HD + (size_t)g * HD;
    const bf16* vg = p.v + ((size_t)b * W + j0) * NKV * HD + (size_t)g * HD;
    bf16* dst = kvb + (c & 1) * 2 * KP * RS;
#pragma unroll
    for (int u = 0; u < 2 * KP * RV / NT; ++u) {
      const int i = tid + u * NT;
      const int r = i / RV, cc = i % RV;
      const int j = r < KP ? r : r - KP;
      const bool ok = j < nk;
      const bf16* src = (r < KP ? kg : vg) + (size_t)(ok ? j : 0) * NKV * HD + cc * 8;
      cp16(dst + r * RS + cc * 8, src, ok);
    }
    cp_commit();
  };

  const int c0 = split * cpc;
  load_chunk(c0);
  {  // the group's 8 query rows (+ 8 zero rows) and zero probability rows 8..15
    const uint4 zero = make_uint4(0, 0, 0, 0);
    const int r = tid / RV, cc = tid % RV;  // 256 threads: 16 rows x 16 pieces
    *reinterpret_cast<uint4*>(qs + r * RS + cc * 8) =
        r < GQ ? __ldg(reinterpret_cast<const uint4*>(p.q + ((size_t)b * NH + (size_t)g * GQ + r) * HD) + cc) : zero;
    if (tid < 8 * (KP / 8)) *reinterpret_cast<uint4*>(ps + (8 + tid / (KP / 8)) * PS + (tid % (KP / 8)) * 8) = zero;
  }

  const int row = lane >> 2;          // query head within the group (C-fragment rows 0..7)
  const int cq = 2 * (lane & 3);      // C-fragment column pair
  const int q8 = lane >> 3;
  float m_run = -INFINITY, l_run = 0.f;
  float o[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
  for (int c = c0; c < c0 + cpc; ++c) {
    if (c + 1 < c0 + cpc) {
      load_chunk(c + 1);
      cp_wait<1>();  // chunk c has landed (this thread's copies)
    } else {
      cp_wait<0>();
    }
    __syncthreads();  // every thread's copies of chunk c (and, first time, the query rows)
    const int j0 = c * CH;
    const int nk = n - j0 < 0 ? 0 : (n - j0 < CH ? n - j0 : CH);
    const bf16* kb_ = kvb + (c & 1) * 2 * KP * RS;
    const bf16* vb_ = kb_ + KP * RS;
    // ---- S = Q K^T: warp w, slots [8w, 8w + 8)
    float sacc[4] = {0.f, 0.f, 0.f, 0.f};
    {
      const uint32_t qb = smem_u32(qs), kb = smem_u32(kb_);
#pragma unroll
      for (int k0 = 0; k0 < HD; k0 += 32) {
        uint32_t a0[4], a1[4], bb[4];
        frag_a(qb, RS, k0, a0);
        frag_a(qb, RS, k0 + 16, a1);
        ldsm_x4(kb + uint32_t(((warp * 8 + (lane & 7)) * RS + k0 + q8 * 8) * 2), bb);
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
    if ((lane & 3) == 0) red[warp * 8 + row] = mw;
    __syncthreads();
    float mc = red[row];
#pragma unroll
    for (int w = 1; w < GQ; ++w) mc = fmaxf(mc, red[w * 8 + row]);
    const float m_new = fmaxf(m_run, mc);
    // a chunk without valid slots leaves everything as it is (m_new may still be -inf)
    const float alpha = m_new == -INFINITY ? 1.f : expf(m_run - m_new);
    const float p0 = jA < nk ? expf(s0 - m_new) : 0.f;
    const float p1 = jA + 1 < nk ? expf(s1 - m_new) : 0.f;
    float lw = p0 + p1;
    lw += __shfl_xor_sync(0xffffffffu, lw, 1);
    lw += __shfl_xor_sync(0xffffffffu, lw, 2);
    if ((lane & 3) == 0) red[GQ * 8 + warp * 8 + row] = lw;
    *reinterpret_cast<__nv_bfloat162*>(ps + row * PS + jA) = __floats2bfloat162_rn(p0, p1);
    __syncthreads();
    float lc = 0.f;
#pragma unroll
    for (int w = 0; w < GQ; ++w) lc += red[GQ * 8 + w * 8 + row];
    l_run = l_run * alpha + lc;
    m_run = m_new;
#pragma unroll
    for (int t = 0; t < 2; ++t)
#pragma unroll
      for (int r = 0; r < 4; ++r) o[t][r] *= alpha;  // rows 8..15 (r >= 2) are zero anyway
    // ---- O += P V: warp w, dimensions [16w, 16w + 16)
    {
      const uint32_t pb0 = smem_u32(ps), vb = smem_u32(vb_);
#pragma unroll
      for (int k0 = 0; k0 < KP; k0 += 32) {
        uint32_t a0[4], a1[4];
        frag_a(pb0, PS, k0, a0);
        frag_a(pb0, PS, k0 + 16, a1);
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          uint32_t bb[4];
          ldsm_x4_t(vb + uint32_t(((k0 + q8 * 8 + (lane & 7)) * RS + warp * 16 + t * 8) * 2), bb);
          mma16816(o[t], a0, bb[0], bb[1]);
          mma16816(o[t], a1, bb[2], bb[3]);
        }
      }
    }
    __syncthreads();  // P, the reductions and this chunk's buffer are free for the next chunk
  }

  const int h = g * GQ + row;
  if (nsplit == 1) {  // the whole window: the output with the sink
    const float sink = __ldg(p.sinks + h);
    const float M = fmaxf(m_run, sink);
    const float a = m_run == -INFINITY ? 0.f : expf(m_run - M);
    const float inv = 1.0f / (l_run * a + expf(sink - M));
#pragma unroll
    for (int t = 0; t < 2; ++t)
      *reinterpret_cast<__nv_bfloat162*>(p.out + ((size_t)b * NH + h) * HD + warp * 16 + t * 8 + cq) =
          __floats2bfloat162_rn(o[t][0] * a * inv, o[t][1] * a * inv);
    return;
  }

  // ---- several splits: the split's partials (o unnormalised, fp32; m; l) per query head
  float* pp = p.part + (((size_t)b * NH + h) * NSPLIT + split) * PSTRIDE;
#pragma unroll
  for (int t = 0; t < 2; ++t)
    *reinterpret_cast<float2*>(pp + warp * 16 + t * 8 + cq) = make_float2(o[t][0], o[t][1]);
  if (warp == 0 && (lane & 3) == 0) {
    pp[HD] = m_run;  // -inf for a split without valid slots (then l = 0 and o = 0)
    pp[HD + 1] = l_run;
  }

  // the last of the splits of (b, g) merges them with the sink (warp w: head 8g + w, lane:
  // dimensions 4 lane .. 4 lane + 3), in split order
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    uint32_t* tk = p.ticket + (size_t)b * NKV + g;
    const uint32_t prev = atomicAdd(tk, 1u);
    s_last = prev == uint32_t(nsplit - 1);
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
    ms[c] = c < nsplit ? __ldcg(ph + c * PSTRIDE + HD) : -INFINITY;
    M = fmaxf(M, ms[c]);
  }
  float L = expf(sink - M);
  float O[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int c = 0; c < NSPLIT; ++c) {
    if (c >= nsplit) break;
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
