// Shared device helpers of the Flint MoE kernels: layer constants, workspace view,
// inline-PTX wrappers (mbarrier, TMA bulk / tensor copies, L2 bulk prefetch, programmatic
// dependent launch) and bounded waits.  sm_103a only.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace flint {

// ---- the only supported layer shape (Flint serving-kit post, "The architecture, from the
// config": hidden 2048, 256 routed experts, 6 per token, widths 512 / 1024)
constexpr int H = 2048;
constexpr int E = 256;
constexpr int K = 6;
constexpr int I = 512;
constexpr int IS = 1024;
// The dense SwiGLU MLP layers before the MoE layers (serving-kit post, "The architecture, from
// the config": mlp_only_layers [0, 1], about 75M parameters for the two) have this width:
// 2 layers x 3 x 2048 x 6144 = 75.5M.  A dense layer runs as the shared-expert path alone.
constexpr int ID = 6144;

using bf16 = __nv_bfloat16;

// ---- device status word bits
constexpr uint32_t ST_TIMEOUT = 1u;
constexpr uint32_t ST_BOUNDS = 2u;

// A bounded wait gives up after this long and records ST_TIMEOUT.
constexpr unsigned long long WAIT_LIMIT_NS = 1000000000ull;  // 1 s

// ---- launch-time parameters shared by every kernel of one forward call
struct Params {
  int T;                 // tokens in this call
  unsigned flags;        // FLINT_MOE_FLAG_*
  float rms_eps;
  int sw;                // width of the shared expert: IS, or ID for a dense MLP layer
  int dense;             // 1: a dense SwiGLU MLP layer (the shared-expert path alone; y = MLP(x') [+ x])
  int fp4;               // 1: NVFP4 expert weights (decode sizes, T <= FP4_MAX_T)
  const float* ts_gate;  // [E] fp32 tensor scales of the routed NVFP4 matrices (fp4)
  const float* ts_up;
  const float* ts_down;
  float ts_sgate, ts_sup, ts_sdown;  // the shared expert's (fp4)
  const uint8_t* q_down;   // [E][I][H/2] routed down codes (fp4; L2 prefetch of the touched experts)
  const uint8_t* q_sdown;  // [IS][H/2] shared down codes (fp4; L2 prefetch)
  const void* fp4_maps;    // the NVFP4 tensor maps (an Fp4Maps in the workspace; fp4)
  const bf16* x;         // layer input [T][H]
  const bf16* xin;       // expert / router input: x, or rms(x) in xn
  bf16* y;               // output [T][H]
  const bf16* w_router;  // [H][E]
  const float* router_bias;  // [E] or null
  const bf16* w_gate;    // [E][H][I]
  const bf16* w_up;      // [E][H][I]
  const bf16* w_down;    // [E][I][H]
  const bf16* ws_gate;   // [H][sw]
  const bf16* ws_up;     // [H][sw]
  const bf16* ws_down;   // [sw][H]
  // workspace
  uint32_t* status;      // [1] device status word (ST_* bits)
  int32_t* counts;       // [E]
  int32_t* offsets;      // [E+1]
  int32_t* perm;         // [T*K] sorted row -> pair (t*K + j)
  int32_t* inv;          // [T*K] pair -> sorted row
  int32_t* topk_idx;     // [T*K]
  float* topk_w;         // [T*K]
  bf16* xn;              // [T][H] rms-normalised input
  bf16* h;               // [T*K][I] routed SwiGLU activations, expert-sorted rows
  bf16* hs;              // [T][sw] shared SwiGLU activations
  float* Y;              // [T*K][H] gated routed expert outputs
  float* S;              // [T][H] shared expert output
  float* P;              // [2 steps][MAX_STREAM_CTAS][2][PSLOT] split-item partial sums (decode path)
  float* RP;             // [32][256][E] router partial logits (decode path)
  bf16* xs;              // [T*K][H] expert-sorted input rows (prefill path)
  bf16* Yb;              // [T*K][H] gated routed expert outputs, bf16 (prefill path)
  int32_t* hist;         // [T/128][E] per-tile expert histogram (prefill path)
  int32_t* mtp;          // [E+1] prefix over experts of their 256-row groups (prefill path)
  uint32_t* bar_count;   // [1] grid-barrier counter (decode path; reset at kernel end)
  uint32_t* bar_done;    // [1]
  uint32_t* tk_gu;       // item tickets (zero between kernels: the last arriver resets)
  uint32_t* tk_sgu;
  uint32_t* tk_sd;
  uint32_t* tk_dn;
  uint32_t* tk_comb;     // [H/128] down items finished per 128-column block (decode path)
  uint32_t* hdone;       // [routed groups] gate/up items finished per routed token group (decode path)
  uint32_t* hsdone;      // [shared groups] shared gate/up items finished per token group (decode path)
  // user-visible copies (may be null)
  int32_t* out_idx;
  float* out_w;
  int32_t* out_counts;
  unsigned long long* trace;  // [gridDim.x][TRACE_SLOTS] %globaltimer stamps, or null
};

constexpr int TRACE_SLOTS = 24;

// Phase trace: thread 0 of each CTA stamps slot `s` with the global timer (ns).
__device__ __forceinline__ void trace_point(const Params& p, int s) {
  if (p.trace && threadIdx.x == 0) {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    p.trace[blockIdx.x * TRACE_SLOTS + s] = t;
  }
}

// ------------------------------------------------------------------ small PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ void record_status(uint32_t* status, uint32_t bit) {
  if (status) atomicOr(status, bit);
}

// Wait for phase `parity` of an mbarrier, giving up after WAIT_LIMIT_NS.  Returns false
// (and records ST_TIMEOUT) when the limit ran out.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint32_t* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > WAIT_LIMIT_NS) {
      record_status(status, ST_TIMEOUT);
      return false;
    }
  }
  return true;
}

// FLINT_MOE_FLAG_TEST_WAIT_TIMEOUT (tests of the device-timeout path only): one thread waits
// for a workspace word that nothing ever writes (status[1]), gives up after a quarter of the
// wait limit -- shorter than every other bounded wait, so the rest of the call proceeds
// normally -- and records ST_TIMEOUT.
constexpr unsigned FLAG_TEST_WAIT_TIMEOUT = 0x80000000u;
__device__ __forceinline__ void test_wait_timeout(uint32_t* status) {
  const volatile uint32_t* never = status + 1;
  const uint64_t t0 = globaltimer_ns();
  while (*never == 0u) {
    if (globaltimer_ns() - t0 > WAIT_LIMIT_NS / 4) {
      record_status(status, ST_TIMEOUT);
      return;
    }
  }
}

// 1-D bulk copy global -> shared (both 16-byte aligned, bytes a multiple of 16), completing
// `bytes` transaction bytes on `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// cp.async of 16 bytes global -> shared, zero-filled when !valid (src_size 0).
__device__ __forceinline__ void cp16(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// 2-D tiled TMA load of box (x = inner coordinate, y = row) into shared memory.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// 3-D tiled TMA load (x = innermost coordinate).
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Ask the memory system to bring `bytes` (multiple of 16) at `src` into L2.
__device__ __forceinline__ void prefetch_l2_bulk(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Programmatic dependent launch: wait for the preceding grid's results / let the next
// grid start launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" :::); }

__device__ __forceinline__ void bf16x8_to_f32(const uint4 v, float* f) {
  f[0] = __uint_as_float(v.x << 16);
  f[1] = __uint_as_float(v.x & 0xFFFF0000u);
  f[2] = __uint_as_float(v.y << 16);
  f[3] = __uint_as_float(v.y & 0xFFFF0000u);
  f[4] = __uint_as_float(v.z << 16);
  f[5] = __uint_as_float(v.z & 0xFFFF0000u);
  f[6] = __uint_as_float(v.w << 16);
  f[7] = __uint_as_float(v.w & 0xFFFF0000u);
}

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) { return __uint_as_float(uint32_t(b) << 16); }

__device__ __forceinline__ float silu_f32(float z) { return z / (1.0f + expf(-z)); }

// silu with the hardware exponential and approximate division (a few ulp in fp32, far below
// the bf16 rounding of the result); for the tensor-core epilogues, whose time per tile is
// bounded by the MMA time of the next tile.  z < -87 gives -0 / +inf -> 0.
__device__ __forceinline__ float silu_fast(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

}  // namespace flint
