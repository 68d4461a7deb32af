// C-ABI of the Flint MoE layer: argument checks, workspace carving, TMA descriptors and the
// launch sequence of each call.  Every step of the layer runs in the kernels included below.
#include <cudaTypedefs.h>

#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "../../include/flint_moe.h"
#include "common.cuh"
#include "decode_fused.cuh"
#include "prefill_kernels.cuh"
#include "swa_attention.cuh"

using namespace flint;

static_assert(FLINT_MOE_FLAG_TEST_WAIT_TIMEOUT == flint::FLAG_TEST_WAIT_TIMEOUT, "flag value");

namespace {

constexpr int MAX_TOKENS_LIMIT = 65536;
constexpr int MAX_EVENTS = 16;
constexpr int MAX_TRACE_CTAS = 1024;

struct Layout {
  // tickets first: [status, tickets) and [tickets, scalars) are cleared together after errors
  size_t status, bar_count, bar_done, tk_gu, tk_sgu, tk_sd, tk_dn, tk_comb, hdone, hsdone;
  size_t zero_end;  // [0, zero_end): status word, barrier counters and tickets (cleared between uses)
  size_t counts, offsets, perm, inv, topk_idx, topk_w;
  size_t xn, xstage, ystage, h, hs, S, Y, P, RP, trace;
  size_t xs, Yb, hist, mtp;  // prefill path (max_tokens > STREAM_MAX_T), else 0
  size_t fp4maps;            // the NVFP4 tensor maps of a handle on NVFP4 weights
  size_t total;
};

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// sw: the shared expert's width (IS), or a dense layer's (ID, with dense = true: no routed
// scratch).
Layout make_layout(int max_tokens, int sw = IS, bool dense = false) {
  Layout L{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = align_up(off, 256);
    off = o + bytes;
    return o;
  };
  const size_t T = (size_t)max_tokens;
  const int Ts = max_tokens < STREAM_MAX_T ? max_tokens : STREAM_MAX_T;
  const size_t G = (size_t)max_groups_upto(Ts);          // routed token groups
  const size_t Gs = (size_t)max_shared_groups_upto(Ts);  // shared token groups
  L.status = take(256);
  L.bar_count = take(sizeof(uint32_t));
  L.bar_done = take(sizeof(uint32_t));
  L.tk_gu = take(sizeof(uint32_t) * G * GU_NCB);
  L.tk_sgu = take(sizeof(uint32_t) * Gs * (sw / 128));
  L.tk_sd = take(sizeof(uint32_t) * Gs * OUT_NCB);
  L.tk_dn = take(sizeof(uint32_t) * G * OUT_NCB);
  L.tk_comb = take(sizeof(uint32_t) * OUT_NCB);
  L.hdone = take(sizeof(uint32_t) * G);
  L.hsdone = take(sizeof(uint32_t) * Gs);
  L.zero_end = align_up(off, 256);
  L.counts = take(sizeof(int32_t) * E);
  L.offsets = take(sizeof(int32_t) * (E + 1));
  L.perm = take(sizeof(int32_t) * T * K);
  L.inv = take(sizeof(int32_t) * T * K);
  L.topk_idx = take(sizeof(int32_t) * T * K);
  L.topk_w = take(sizeof(float) * T * K);
  L.xn = take(sizeof(uint16_t) * T * H);
  L.xstage = take(sizeof(uint16_t) * T * H);
  L.ystage = take(sizeof(uint16_t) * T * H);
  L.h = take(sizeof(uint16_t) * T * K * I);
  L.hs = take(sizeof(uint16_t) * T * sw);
  L.S = take(sizeof(float) * T * H);
  L.Y = take(sizeof(float) * (size_t)Ts * K * H);
  L.P = take(sizeof(float) * 2 * MAX_STREAM_CTAS * 2 * PSLOT);  // two banks: steps C and D
  L.RP = take(sizeof(float) * RT_NB * STREAM_MAX_T * E);
  if (max_tokens > STREAM_MAX_T && !dense) {
    const size_t ntile = (T + tc::TM - 1) / tc::TM;
    L.xs = take(sizeof(uint16_t) * T * K * H);
    L.Yb = take(sizeof(uint16_t) * T * K * H);
    L.hist = take(sizeof(int32_t) * ntile * E);
    L.mtp = take(sizeof(int32_t) * (E + 1));
  }
  L.trace = take(sizeof(unsigned long long) * MAX_TRACE_CTAS * TRACE_SLOTS);
  L.fp4maps = take(sizeof(Fp4Maps));
  L.total = align_up(off, 256);
  return L;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* ptr = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// Row-major bf16 matrix [rows][cols] -> 2-D tensor map with a box of box_cols x box_rows.  L2
// fills are promoted to 128 bytes only: a box row is 128 bytes, and a wider promotion would
// fetch the neighbouring columns, which are read much later (by then evicted) when the stream
// is larger than L2.
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_cols,
              uint32_t box_rows, CUtensorMapSwizzle swz) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// K-major NVFP4 gate/up codes [rows][1024 bytes] as a 3-D tensor (128 bytes of a row, rows, the row's
// eight 128-byte pieces): a box of 128 x 16 rows x 8 pieces is 16 whole rows (16 KB, contiguous in
// memory), laid out in shared memory as [piece][row][128 bytes] with the 128-byte swizzle.
bool make_map_fp4_rows(CUtensorMap* m, const void* base, uint64_t rows) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {128, rows, 8};
  cuuint64_t strides[2] = {1024, 128};
  cuuint32_t box[3] = {128, 16, 8};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Row-major uint8 matrix [rows][cols] (NVFP4 codes or scales) -> 2-D tensor map, box of box_cols
// bytes x box_rows (codes: 128-byte rows with the 128-byte swizzle; scales: no swizzle).
bool make_map_u8(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_cols,
                 uint32_t box_rows, CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_NONE) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace

struct flint_moe_stack_s {
  flint_moe_t h;    // handle on layer 0's weights and the shared scratch
  int n_layers;
  void* tab;        // device table of LayerTab entries (in the workspace)
};

struct flint_moe_s {
  flint_moe_config cfg;
  flint_moe_weights w;
  int sw;      // the shared expert's width (IS), or the dense layer's (ID)
  int dense;   // 1: a dense SwiGLU MLP layer (flint_dense_*): the shared-expert path alone
  int fp4;     // 1: NVFP4 expert weights (flint_moe_create_nvfp4)
  flint_moe_nvfp4_weights q;  // the NVFP4 weights (fp4)
  int device;
  int n_sm;
  uint8_t* ws;
  size_t ws_bytes;
  Layout L;
  StreamMaps smaps;
  pf::Maps pmaps;  // prefill path (max_tokens > STREAM_MAX_T); pmaps.xin is on xn
  bool timing;
  bool trace;
  cudaEvent_t ev[2 * MAX_EVENTS];
  const char* ev_name[MAX_EVENTS];
  int n_ev;
};

namespace {

flint_moe_status check_config(const flint_moe_config* c) {
  if (!c) return FLINT_MOE_ERR_INVALID_ARG;
  if (c->hidden != H || c->n_experts != E || c->top_k != K || c->expert_inter != I || c->shared_inter != IS)
    return FLINT_MOE_ERR_UNSUPPORTED;
  if (c->max_tokens < 1 || c->max_tokens > MAX_TOKENS_LIMIT) return FLINT_MOE_ERR_INVALID_ARG;
  if (c->flags & ~(FLINT_MOE_FLAG_PRE_RMSNORM | FLINT_MOE_FLAG_RESIDUAL | FLINT_MOE_FLAG_TEST_WAIT_TIMEOUT))
    return FLINT_MOE_ERR_UNSUPPORTED;
  if ((c->flags & FLINT_MOE_FLAG_PRE_RMSNORM) && !(c->rms_eps > 0.f)) return FLINT_MOE_ERR_INVALID_ARG;
  return FLINT_MOE_OK;
}

Params make_params(flint_moe_t h, const void* x, int T, void* y, int32_t* out_idx, float* out_w,
                   int32_t* out_counts) {
  Params p{};
  uint8_t* ws = h->ws;
  const Layout& L = h->L;
  p.T = T;
  p.flags = h->cfg.flags;
  p.rms_eps = h->cfg.rms_eps;
  p.sw = h->sw;
  p.dense = h->dense;
  p.fp4 = h->fp4;
  if (h->fp4) {
    p.ts_gate = h->q.gate_tscale;
    p.ts_up = h->q.up_tscale;
    p.ts_down = h->q.down_tscale;
    p.ts_sgate = h->q.sgate_tscale;
    p.ts_sup = h->q.sup_tscale;
    p.ts_sdown = h->q.sdown_tscale;
    p.q_down = h->q.down_codes;
    p.q_sdown = h->q.sdown_codes;
    p.fp4_maps = ws + L.fp4maps;
  }
  p.x = static_cast<const bf16*>(x);
  p.xn = reinterpret_cast<bf16*>(ws + L.xn);
  p.xin = (h->cfg.flags & FLINT_MOE_FLAG_PRE_RMSNORM) ? p.xn : p.x;
  p.y = static_cast<bf16*>(y);
  p.w_router = static_cast<const bf16*>(h->w.w_router);
  p.router_bias = h->w.router_bias;
  p.w_gate = static_cast<const bf16*>(h->w.w_gate);
  p.w_up = static_cast<const bf16*>(h->w.w_up);
  p.w_down = static_cast<const bf16*>(h->w.w_down);
  p.ws_gate = static_cast<const bf16*>(h->w.ws_gate);
  p.ws_up = static_cast<const bf16*>(h->w.ws_up);
  p.ws_down = static_cast<const bf16*>(h->w.ws_down);
  p.status = reinterpret_cast<uint32_t*>(ws + L.status);
  p.bar_count = reinterpret_cast<uint32_t*>(ws + L.bar_count);
  p.bar_done = reinterpret_cast<uint32_t*>(ws + L.bar_done);
  p.tk_gu = reinterpret_cast<uint32_t*>(ws + L.tk_gu);
  p.tk_sgu = reinterpret_cast<uint32_t*>(ws + L.tk_sgu);
  p.tk_sd = reinterpret_cast<uint32_t*>(ws + L.tk_sd);
  p.tk_dn = reinterpret_cast<uint32_t*>(ws + L.tk_dn);
  p.tk_comb = reinterpret_cast<uint32_t*>(ws + L.tk_comb);
  p.hdone = reinterpret_cast<uint32_t*>(ws + L.hdone);
  p.hsdone = reinterpret_cast<uint32_t*>(ws + L.hsdone);
  p.counts = reinterpret_cast<int32_t*>(ws + L.counts);
  p.offsets = reinterpret_cast<int32_t*>(ws + L.offsets);
  p.perm = reinterpret_cast<int32_t*>(ws + L.perm);
  p.inv = reinterpret_cast<int32_t*>(ws + L.inv);
  p.topk_idx = reinterpret_cast<int32_t*>(ws + L.topk_idx);
  p.topk_w = reinterpret_cast<float*>(ws + L.topk_w);
  p.h = reinterpret_cast<bf16*>(ws + L.h);
  p.hs = reinterpret_cast<bf16*>(ws + L.hs);
  p.S = reinterpret_cast<float*>(ws + L.S);
  p.Y = reinterpret_cast<float*>(ws + L.Y);
  p.P = reinterpret_cast<float*>(ws + L.P);
  p.RP = reinterpret_cast<float*>(ws + L.RP);
  if (L.Yb) {
    p.xs = reinterpret_cast<bf16*>(ws + L.xs);
    p.Yb = reinterpret_cast<bf16*>(ws + L.Yb);
    p.hist = reinterpret_cast<int32_t*>(ws + L.hist);
    p.mtp = reinterpret_cast<int32_t*>(ws + L.mtp);
  }
  p.out_idx = out_idx;
  p.out_w = out_w;
  p.out_counts = out_counts;
  p.trace = h->trace ? reinterpret_cast<unsigned long long*>(ws + L.trace) : nullptr;
  return p;
}

// Launch with programmatic stream serialisation, or as a cooperative grid (all CTAs
// resident at once, required by kernels with grid-wide barriers).
template <class... KArgs, class... Args>
cudaError_t launch(flint_moe_t h, const char* name, void (*kern)(KArgs...), unsigned grid, unsigned block, int smem,
                   cudaStream_t st, bool cooperative, Args&&... args) {
  if (grid == 0) return cudaSuccess;
  const bool rec = h->timing && h->n_ev < MAX_EVENTS;
  if (rec) {
    h->ev_name[h->n_ev] = name;
    cudaEventRecord(h->ev[2 * h->n_ev], st);
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  if (cooperative) {
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
  } else {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
  }
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
  if (rec) {
    cudaEventRecord(h->ev[2 * h->n_ev + 1], st);
    h->n_ev++;
  }
  return e;
}

// The layer on T <= STREAM_MAX_T tokens (weights described by `maps` and p): optional RMSNorm
// kernel, then the persistent cooperative decode kernel (one CTA per SM).
flint_moe_status run_decode_maps(flint_moe_t h, const Params& p, const StreamMaps& maps, cudaStream_t st,
                                 bool full) {
  cudaError_t e = cudaSuccess;
  if (h->cfg.flags & FLINT_MOE_FLAG_PRE_RMSNORM) e = launch(h, "rmsnorm", rmsnorm_kernel, p.T, 256, 0, st, false, p);
  if (e != cudaSuccess) return FLINT_MOE_ERR_CUDA;
  const int grid = h->n_sm < MAX_STREAM_CTAS ? h->n_sm : MAX_STREAM_CTAS;
  auto kern = h->fp4 ? decode_fused<MODE_FP4> : h->dense ? decode_fused<MODE_DENSE> : decode_fused<MODE_MOE>;
  e = launch(h, full ? "decode_fused" : "decode_fused_route", kern, grid, NTHREADS,
             h->fp4 ? fp4_smem_bytes() : fused_smem_bytes(group_rows_mode(p.T, h->dense ? MODE_DENSE : MODE_MOE)), st, true, p, maps, full ? 0 : 1);
  return e == cudaSuccess ? FLINT_MOE_OK : FLINT_MOE_ERR_CUDA;
}

flint_moe_status run_decode(flint_moe_t h, const Params& p, cudaStream_t st, bool full) {
  return run_decode_maps(h, p, h->smaps, st, full);
}

// The layer on T > STREAM_MAX_T tokens: the tensor-core path (prefill_kernels.cuh), five (six
// with pre-norm) stream-ordered kernels with programmatic dependent launch.
flint_moe_status run_prefill(flint_moe_t h, const Params& p, cudaStream_t st, bool full) {
  const int T = p.T;
  const int ntile = (T + tc::TM - 1) / tc::TM;
  cudaError_t e = cudaSuccess;
  if (h->cfg.flags & FLINT_MOE_FLAG_PRE_RMSNORM) e = launch(h, "rmsnorm", rmsnorm_kernel, T, 256, 0, st, false, p);
  if (e != cudaSuccess) return FLINT_MOE_ERR_CUDA;
  // the A operand of the router and of the shared gate/up: the layer input rows
  CUtensorMap xin = h->pmaps.xin, xin_c = h->pmaps.xin_c;
  if (!(h->cfg.flags & FLINT_MOE_FLAG_PRE_RMSNORM) &&
      !(make_map(&xin, p.x, (uint64_t)T, H, 64, tc::TM, CU_TENSOR_MAP_SWIZZLE_128B) &&
        make_map(&xin_c, p.x, (uint64_t)T, H, 64, tc::XC_ROWS, CU_TENSOR_MAP_SWIZZLE_128B)))
    return FLINT_MOE_ERR_CUDA;
  const int n_sm = h->n_sm;
  if (h->dense) {  // the shared-expert GEMMs alone; the down epilogue writes y
    pf::GateUpTC gu{p, h->pmaps.xs, xin_c, h->pmaps.wg, h->pmaps.wu, h->pmaps.wsg, h->pmaps.wsu};
    e = launch(h, "pf_gateup", tc::gemm_kernel<pf::GateUpTC>, n_sm, tc::NUM_THREADS, tc::SMEM_BYTES, st, false, gu);
    pf::DownTC dn{p, h->pmaps.h, h->pmaps.wd, h->pmaps.hs, h->pmaps.wsd};
    if (e == cudaSuccess)
      e = launch(h, "pf_down", tc::gemm_kernel<pf::DownTC>, n_sm, tc::NUM_THREADS, tc::SMEM_BYTES, st, false, dn);
    return e == cudaSuccess ? FLINT_MOE_OK : FLINT_MOE_ERR_CUDA;
  }
  pf::RouterTC r{p, xin, h->pmaps.wr};
  e = launch(h, "pf_router", tc::gemm_kernel<pf::RouterTC>, ntile < n_sm ? ntile : n_sm, tc::NUM_THREADS,
             tc::SMEM_BYTES, st, false, r);
  if (e != cudaSuccess) return FLINT_MOE_ERR_CUDA;
  if (!full) {
    e = launch(h, "pf_scatter", pf::scatter_kernel, 1, 256, 0, st, false, p, 0);
    return e == cudaSuccess ? FLINT_MOE_OK : FLINT_MOE_ERR_CUDA;
  }
  e = launch(h, "pf_scatter", pf::scatter_kernel, ntile * pf::SPLIT, 256, 0, st, false, p, 1);
  pf::GateUpTC gu{p, h->pmaps.xs, xin_c, h->pmaps.wg, h->pmaps.wu, h->pmaps.wsg, h->pmaps.wsu};
  if (e == cudaSuccess)
    e = launch(h, "pf_gateup", tc::gemm_kernel<pf::GateUpTC>, n_sm, tc::NUM_THREADS, tc::SMEM_BYTES, st, false, gu);
  pf::DownTC dn{p, h->pmaps.h, h->pmaps.wd, h->pmaps.hs, h->pmaps.wsd};
  if (e == cudaSuccess)
    e = launch(h, "pf_down", tc::gemm_kernel<pf::DownTC>, n_sm, tc::NUM_THREADS, tc::SMEM_BYTES, st, false, dn);
  if (e == cudaSuccess) e = launch(h, "pf_combine", pf::combine_kernel, T, 256, 0, st, false, p);
  return e == cudaSuccess ? FLINT_MOE_OK : FLINT_MOE_ERR_CUDA;
}

flint_moe_status run_layer(flint_moe_t h, const Params& p, cudaStream_t st, bool full) {
  // a traced call starts from a cleared trace: slots that its kernels do not stamp read 0
  if (p.trace && cudaMemsetAsync(p.trace, 0, sizeof(unsigned long long) * MAX_TRACE_CTAS * TRACE_SLOTS, st) !=
                     cudaSuccess)
    return FLINT_MOE_ERR_CUDA;
  return p.T <= STREAM_MAX_T ? run_decode(h, p, st, full) : run_prefill(h, p, st, full);
}

flint_moe_status check_call(flint_moe_t h, const void* x, int T) {
  if (!h) return FLINT_MOE_ERR_INVALID_ARG;
  if (!x || !aligned16(x)) return FLINT_MOE_ERR_INVALID_ARG;
  if (T < 1 || T > h->cfg.max_tokens) return FLINT_MOE_ERR_INVALID_ARG;
  return FLINT_MOE_OK;
}

// Tensor maps of the prefill path (weights: boxes of 64 x 64; activations read by the router's
// ROWS tiles: boxes of 64 x 128; activations read by COLUMNS tiles: boxes of 64 x 64).  Needs
// the workspace carved (h->ws, h->L).
bool make_prefill_maps(flint_moe_t h) {
  const auto sw = CU_TENSOR_MAP_SWIZZLE_128B;
  const flint_moe_weights* w = &h->w;
  const uint64_t T = (uint64_t)h->cfg.max_tokens;
  pf::Maps& m = h->pmaps;
  const uint64_t S = (uint64_t)h->sw;
  if (h->dense)
    return make_map(&m.xin, h->ws + h->L.xn, T, H, 64, tc::TM, sw) &&
           make_map(&m.xin_c, h->ws + h->L.xn, T, H, 64, tc::XC_ROWS, sw) &&
           make_map(&m.hs, h->ws + h->L.hs, T, S, 64, tc::XC_ROWS, sw) &&
           make_map(&m.wsg, w->ws_gate, H, S, 64, tc::TK, sw) && make_map(&m.wsu, w->ws_up, H, S, 64, tc::TK, sw) &&
           make_map(&m.wsd, w->ws_down, S, H, 64, tc::TK, sw);
  return make_map(&m.xin, h->ws + h->L.xn, T, H, 64, tc::TM, sw) &&
         make_map(&m.xin_c, h->ws + h->L.xn, T, H, 64, tc::XC_ROWS, sw) &&
         make_map(&m.xs, h->ws + h->L.xs, T * K, H, 64, tc::XC_ROWS, sw) &&
         make_map(&m.h, h->ws + h->L.h, T * K, I, 64, tc::XC_ROWS, sw) &&
         make_map(&m.hs, h->ws + h->L.hs, T, IS, 64, tc::XC_ROWS, sw) &&
         make_map(&m.wr, w->w_router, H, E, 64, tc::TK, sw) &&
         make_map(&m.wg, w->w_gate, (uint64_t)E * H, I, 64, tc::TK, sw) &&
         make_map(&m.wu, w->w_up, (uint64_t)E * H, I, 64, tc::TK, sw) &&
         make_map(&m.wd, w->w_down, (uint64_t)E * I, H, 64, tc::TK, sw) &&
         make_map(&m.wsg, w->ws_gate, H, IS, 64, tc::TK, sw) &&
         make_map(&m.wsu, w->ws_up, H, IS, 64, tc::TK, sw) &&
         make_map(&m.wsd, w->ws_down, IS, H, 64, tc::TK, sw);
}

cudaError_t set_prefill_smem() {
  cudaError_t e = cudaFuncSetAttribute(tc::gemm_kernel<pf::RouterTC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       tc::SMEM_BYTES);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(tc::gemm_kernel<pf::GateUpTC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             tc::SMEM_BYTES);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(tc::gemm_kernel<pf::DownTC>, cudaFuncAttributeMaxDynamicSharedMemorySize, tc::SMEM_BYTES);
  return e;
}

}  // namespace

extern "C" {

const char* flint_moe_status_string(flint_moe_status s) {
  switch (s) {
    case FLINT_MOE_OK: return "ok";
    case FLINT_MOE_ERR_INVALID_ARG: return "invalid argument";
    case FLINT_MOE_ERR_UNSUPPORTED: return "unsupported shape, flags or device";
    case FLINT_MOE_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case FLINT_MOE_ERR_CUDA: return "CUDA runtime error";
    case FLINT_MOE_ERR_DEVICE_TIMEOUT: return "a bounded device-side wait ran out";
    case FLINT_MOE_ERR_DEVICE_BOUNDS: return "a device-side index check failed";
  }
  return "unknown status";
}

flint_moe_status flint_moe_workspace_bytes(const flint_moe_config* cfg, size_t* bytes) {
  flint_moe_status s = check_config(cfg);
  if (s != FLINT_MOE_OK) return s;
  if (!bytes) return FLINT_MOE_ERR_INVALID_ARG;
  *bytes = make_layout(cfg->max_tokens).total;
  return FLINT_MOE_OK;
}

}  // extern "C"

namespace {

// A handle on validated arguments: the MoE layer (sw = IS, dense = false; every weight pointer
// set), a dense layer (sw = ID, dense = true; only the shared-expert pointers of `w` are used) or
// an NVFP4 MoE layer (router_only: only the router's maps here; the caller adds the NVFP4 ones).
flint_moe_status create_handle(const flint_moe_config* cfg, const flint_moe_weights* w, void* workspace,
                               size_t workspace_bytes, int swidth, bool dense, flint_moe_t* out,
                               bool router_only = false) {
  Layout L = make_layout(cfg->max_tokens, swidth, dense);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < L.total)
    return FLINT_MOE_ERR_WORKSPACE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FLINT_MOE_ERR_CUDA;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return FLINT_MOE_ERR_CUDA;
  if (major != 10 || minor != 3) return FLINT_MOE_ERR_UNSUPPORTED;

  flint_moe_s* h = new (std::nothrow) flint_moe_s();
  if (!h) return FLINT_MOE_ERR_CUDA;
  h->cfg = *cfg;
  h->w = *w;
  h->sw = swidth;
  h->dense = dense ? 1 : 0;
  h->device = dev;
  h->ws = static_cast<uint8_t*>(workspace);
  h->ws_bytes = workspace_bytes;
  h->L = L;
  h->timing = false;
  h->trace = false;
  h->n_ev = 0;
  if (cudaDeviceGetAttribute(&h->n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || h->n_sm < 1) {
    delete h;
    return FLINT_MOE_ERR_CUDA;
  }
  const auto sw = CU_TENSOR_MAP_SWIZZLE_128B;
  const uint64_t S = (uint64_t)swidth;
  bool ok = router_only ? make_map(&h->smaps.wr, w->w_router, H, E, 64, RT_ROWS, sw)
                        : make_map(&h->smaps.wsg, w->ws_gate, H, S, 64, GU_ROWS, sw) &&
                              make_map(&h->smaps.wsu, w->ws_up, H, S, 64, GU_ROWS, sw) &&
                              make_map(&h->smaps.wsd, w->ws_down, S, H, 64, DN_ROWS, sw);
  if (ok && !dense && !router_only)
    ok = make_map(&h->smaps.wr, w->w_router, H, E, 64, RT_ROWS, sw) &&
         make_map(&h->smaps.wg, w->w_gate, (uint64_t)E * H, I, 64, GU_ROWS, sw) &&
         make_map(&h->smaps.wu, w->w_up, (uint64_t)E * H, I, 64, GU_ROWS, sw) &&
         make_map(&h->smaps.wd, w->w_down, (uint64_t)E * I, H, 64, DN_ROWS, sw);
  const bool prefill = cfg->max_tokens > STREAM_MAX_T;
  if (ok && prefill) ok = make_prefill_maps(h);
  if (!ok) {
    delete h;
    return FLINT_MOE_ERR_CUDA;
  }
  // every mode's instantiation (a handle made here may be turned into an NVFP4 one by the caller)
  cudaError_t e = cudaSuccess;
  for (auto kern : {decode_fused<MODE_MOE>, decode_fused<MODE_FP4>, decode_fused<MODE_DENSE>}) {
    if (e == cudaSuccess) e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, FUSED_SMEM);
    int per_sm = 0;
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, NTHREADS, FUSED_SMEM);
    if (e == cudaSuccess && per_sm < 1) e = cudaErrorCooperativeLaunchTooLarge;
  }
  if (e == cudaSuccess && prefill) e = set_prefill_smem();
  if (e == cudaSuccess) e = cudaMemset(h->ws, 0, L.xn);  // status, tickets and routing scratch
  for (int i = 0; i < 2 * MAX_EVENTS && e == cudaSuccess; ++i) e = cudaEventCreate(&h->ev[i]);
  if (e != cudaSuccess) {
    delete h;
    return FLINT_MOE_ERR_CUDA;
  }
  *out = h;
  return FLINT_MOE_OK;
}

}  // namespace

extern "C" {

flint_moe_status flint_moe_create(const flint_moe_config* cfg, const flint_moe_weights* w, void* workspace,
                                  size_t workspace_bytes, flint_moe_t* out) {
  if (!out) return FLINT_MOE_ERR_INVALID_ARG;
  *out = nullptr;
  flint_moe_status s = check_config(cfg);
  if (s != FLINT_MOE_OK) return s;
  if (!w || !w->w_router || !w->w_gate || !w->w_up || !w->w_down || !w->ws_gate || !w->ws_up || !w->ws_down)
    return FLINT_MOE_ERR_INVALID_ARG;
  const void* ptrs[] = {w->w_router, w->w_gate, w->w_up, w->w_down, w->ws_gate, w->ws_up, w->ws_down};
  for (const void* q : ptrs)
    if (!aligned16(q)) return FLINT_MOE_ERR_INVALID_ARG;
  if (w->router_bias && (reinterpret_cast<uintptr_t>(w->router_bias) & 3u)) return FLINT_MOE_ERR_INVALID_ARG;
  return create_handle(cfg, w, workspace, workspace_bytes, IS, false, out);
}

flint_moe_status flint_moe_route(flint_moe_t h, const void* x, int T, int32_t* topk_idx, float* topk_w,
                                 int32_t* counts, flint_stream_t stream) {
  flint_moe_status s = check_call(h, x, T);
  if (s != FLINT_MOE_OK) return s;
  if (!topk_idx || !topk_w) return FLINT_MOE_ERR_INVALID_ARG;
  h->n_ev = 0;
  Params p = make_params(h, x, T, nullptr, topk_idx, topk_w, counts);
  return run_layer(h, p, reinterpret_cast<cudaStream_t>(stream), false);
}

flint_moe_status flint_moe_forward(flint_moe_t h, const void* x, int T, void* y, int32_t* topk_idx,
                                   float* topk_w, flint_stream_t stream) {
  flint_moe_status s = check_call(h, x, T);
  if (s != FLINT_MOE_OK) return s;
  if (!y || !aligned16(y)) return FLINT_MOE_ERR_INVALID_ARG;
  h->n_ev = 0;
  Params p = make_params(h, x, T, y, topk_idx, topk_w, nullptr);
  return run_layer(h, p, reinterpret_cast<cudaStream_t>(stream), true);
}

flint_moe_status flint_moe_forward_host(flint_moe_t h, const void* x_host, int T, void* y_host,
                                        flint_stream_t stream) {
  if (!h || !x_host || !y_host) return FLINT_MOE_ERR_INVALID_ARG;
  if (T < 1 || T > h->cfg.max_tokens) return FLINT_MOE_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  void* xd = h->ws + h->L.xstage;
  void* yd = h->ws + h->L.ystage;
  const size_t bytes = (size_t)T * H * sizeof(uint16_t);
  if (cudaMemcpyAsync(xd, x_host, bytes, cudaMemcpyHostToDevice, st) != cudaSuccess) return FLINT_MOE_ERR_CUDA;
  flint_moe_status s = flint_moe_forward(h, xd, T, yd, nullptr, nullptr, stream);
  if (s != FLINT_MOE_OK) return s;
  if (cudaMemcpyAsync(y_host, yd, bytes, cudaMemcpyDeviceToHost, st) != cudaSuccess) return FLINT_MOE_ERR_CUDA;
  return FLINT_MOE_OK;
}

flint_moe_status flint_moe_poll_device_status(flint_moe_t h, flint_stream_t stream) {
  if (!h) return FLINT_MOE_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return FLINT_MOE_ERR_CUDA;
  uint32_t word = 0;
  if (cudaMemcpy(&word, h->ws + h->L.status, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess)
    return FLINT_MOE_ERR_CUDA;
  if (word == 0) return FLINT_MOE_OK;
  // A device error may leave tickets mid-count: clear them with the status word.
  if (cudaMemset(h->ws + h->L.status, 0, h->L.zero_end - h->L.status) != cudaSuccess) return FLINT_MOE_ERR_CUDA;
  return (word & ST_TIMEOUT) ? FLINT_MOE_ERR_DEVICE_TIMEOUT : FLINT_MOE_ERR_DEVICE_BOUNDS;
}

flint_moe_status flint_moe_enable_kernel_timing(flint_moe_t h, int enable) {
  if (!h) return FLINT_MOE_ERR_INVALID_ARG;
  h->timing = enable == 1;
  h->trace = enable == 2;
  h->n_ev = 0;
  return FLINT_MOE_OK;
}

flint_moe_status flint_moe_read_trace(flint_moe_t h, unsigned long long* out, int cap, int* n) {
  if (!h || !n || cap < 0 || (cap > 0 && !out)) return FLINT_MOE_ERR_INVALID_ARG;
  const int total = (h->n_sm < MAX_TRACE_CTAS ? h->n_sm : MAX_TRACE_CTAS) * TRACE_SLOTS;
  const int m = total < cap ? total : cap;
  if (cudaDeviceSynchronize() != cudaSuccess) return FLINT_MOE_ERR_CUDA;
  if (m > 0 && cudaMemcpy(out, h->ws + h->L.trace, sizeof(unsigned long long) * m, cudaMemcpyDeviceToHost) !=
                   cudaSuccess)
    return FLINT_MOE_ERR_CUDA;
  *n = m;
  return FLINT_MOE_OK;
}

flint_moe_status flint_moe_kernel_times(flint_moe_t h, const char** names, float* ms, int cap, int* n) {
  if (!h || !n || cap < 0 || (cap > 0 && (!names || !ms))) return FLINT_MOE_ERR_INVALID_ARG;
  int m = h->n_ev < cap ? h->n_ev : cap;
  for (int i = 0; i < m; ++i) {
    if (cudaEventSynchronize(h->ev[2 * i + 1]) != cudaSuccess) return FLINT_MOE_ERR_CUDA;
    float t = 0.f;
    if (cudaEventElapsedTime(&t, h->ev[2 * i], h->ev[2 * i + 1]) != cudaSuccess) return FLINT_MOE_ERR_CUDA;
    names[i] = h->ev_name[i];
    ms[i] = t;
  }
  *n = m;
  return FLINT_MOE_OK;
}

flint_moe_status flint_moe_destroy(flint_moe_t h) {
  if (!h) return FLINT_MOE_ERR_INVALID_ARG;
  for (int i = 0; i < 2 * MAX_EVENTS; ++i)
    if (h->ev[i]) cudaEventDestroy(h->ev[i]);
  delete h;
  return FLINT_MOE_OK;
}

// ---------------------------------------------------------------- the layer stack
// The stack's workspace: the scratch of one layer with max_tokens tokens (its counters,
// tables and intermediates serve every layer in turn), then the device table of per-layer
// tensor maps and weight pointers.
flint_moe_status flint_moe_stack_workspace_bytes(const flint_moe_config* cfg, int n_layers, size_t* bytes) {
  flint_moe_status s = check_config(cfg);
  if (s != FLINT_MOE_OK) return s;
  if (!bytes || n_layers < 1) return FLINT_MOE_ERR_INVALID_ARG;
  if (cfg->max_tokens > STREAM_MAX_T) return FLINT_MOE_ERR_UNSUPPORTED;
  *bytes = align_up(make_layout(cfg->max_tokens).total, 256) + align_up(sizeof(LayerTab) * n_layers, 256);
  return FLINT_MOE_OK;
}

flint_moe_status flint_moe_stack_create(const flint_moe_config* cfg, const flint_moe_weights* layers, int n_layers,
                                        void* workspace, size_t workspace_bytes, flint_moe_stack_t* out) {
  if (!out) return FLINT_MOE_ERR_INVALID_ARG;
  *out = nullptr;
  size_t need = 0;
  flint_moe_status s = flint_moe_stack_workspace_bytes(cfg, n_layers, &need);
  if (s != FLINT_MOE_OK) return s;
  if (!layers) return FLINT_MOE_ERR_INVALID_ARG;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < need)
    return FLINT_MOE_ERR_WORKSPACE;
  for (int l = 0; l < n_layers; ++l) {
    const flint_moe_weights* w = &layers[l];
    if (!w->w_router || !w->w_gate || !w->w_up || !w->w_down || !w->ws_gate || !w->ws_up || !w->ws_down)
      return FLINT_MOE_ERR_INVALID_ARG;
    const void* ptrs[] = {w->w_router, w->w_gate, w->w_up, w->w_down, w->ws_gate, w->ws_up, w->ws_down};
    for (const void* q : ptrs)
      if (!aligned16(q)) return FLINT_MOE_ERR_INVALID_ARG;
    if (w->router_bias && (reinterpret_cast<uintptr_t>(w->router_bias) & 3u)) return FLINT_MOE_ERR_INVALID_ARG;
  }
  const size_t scratch = align_up(make_layout(cfg->max_tokens).total, 256);
  flint_moe_t h = nullptr;
  s = flint_moe_create(cfg, &layers[0], workspace, scratch, &h);
  if (s != FLINT_MOE_OK) return s;
  std::vector<LayerTab> tab(n_layers);
  const auto sw = CU_TENSOR_MAP_SWIZZLE_128B;
  bool ok = true;
  for (int l = 0; l < n_layers && ok; ++l) {
    const flint_moe_weights* w = &layers[l];
    LayerTab& t = tab[l];
    std::memset(&t, 0, sizeof t);
    ok = make_map(&t.maps.wr, w->w_router, H, E, 64, RT_ROWS, sw) &&
         make_map(&t.maps.wg, w->w_gate, (uint64_t)E * H, I, 64, GU_ROWS, sw) &&
         make_map(&t.maps.wu, w->w_up, (uint64_t)E * H, I, 64, GU_ROWS, sw) &&
         make_map(&t.maps.wd, w->w_down, (uint64_t)E * I, H, 64, DN_ROWS, sw) &&
         make_map(&t.maps.wsg, w->ws_gate, H, IS, 64, GU_ROWS, sw) &&
         make_map(&t.maps.wsu, w->ws_up, H, IS, 64, GU_ROWS, sw) &&
         make_map(&t.maps.wsd, w->ws_down, IS, H, 64, DN_ROWS, sw);
    t.router_bias = w->router_bias;
    t.w_router = static_cast<const bf16*>(w->w_router);
    t.ws_gate = static_cast<const bf16*>(w->ws_gate);
    t.ws_up = static_cast<const bf16*>(w->ws_up);
    t.ws_down = static_cast<const bf16*>(w->ws_down);
  }
  LayerTab* dtab = reinterpret_cast<LayerTab*>(static_cast<uint8_t*>(workspace) + scratch);
  cudaError_t e = ok ? cudaSuccess : cudaErrorInvalidValue;
  if (e == cudaSuccess) e = cudaMemcpy(dtab, tab.data(), sizeof(LayerTab) * n_layers, cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(decode_stack, cudaFuncAttributeMaxDynamicSharedMemorySize, FUSED_SMEM);
  int per_sm = 0;
  if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_stack, NTHREADS, FUSED_SMEM);
  if (e == cudaSuccess && per_sm < 1) e = cudaErrorCooperativeLaunchTooLarge;
  flint_moe_stack_s* st = e == cudaSuccess ? new (std::nothrow) flint_moe_stack_s() : nullptr;
  if (!st) {
    flint_moe_destroy(h);
    return FLINT_MOE_ERR_CUDA;
  }
  st->h = h;
  st->n_layers = n_layers;
  st->tab = dtab;
  *out = st;
  return FLINT_MOE_OK;
}

flint_moe_status flint_moe_stack_forward(flint_moe_stack_t st, void* x, int T, int32_t* topk_idx, float* topk_w,
                                         flint_stream_t stream) {
  if (!st) return FLINT_MOE_ERR_INVALID_ARG;
  flint_moe_t h = st->h;
  flint_moe_status s = check_call(h, x, T);
  if (s != FLINT_MOE_OK) return s;
  h->n_ev = 0;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  Params p = make_params(h, x, T, x, topk_idx, topk_w, nullptr);
  if (p.trace && cudaMemsetAsync(p.trace, 0, sizeof(unsigned long long) * MAX_TRACE_CTAS * TRACE_SLOTS, cs) !=
                     cudaSuccess)
    return FLINT_MOE_ERR_CUDA;
  const int grid = h->n_sm < MAX_STREAM_CTAS ? h->n_sm : MAX_STREAM_CTAS;
  const cudaError_t e = launch(h, "decode_stack", decode_stack, grid, NTHREADS, fused_smem_bytes(group_rows(T)), cs, true, p,
                               static_cast<const LayerTab*>(st->tab), st->n_layers);
  return e == cudaSuccess ? FLINT_MOE_OK : FLINT_MOE_ERR_CUDA;
}

flint_moe_status flint_moe_stack_poll_device_status(flint_moe_stack_t st, flint_stream_t stream) {
  if (!st) return FLINT_MOE_ERR_INVALID_ARG;
  return flint_moe_poll_device_status(st->h, stream);
}

flint_moe_status flint_moe_stack_enable_kernel_timing(flint_moe_stack_t st, int enable) {
  if (!st) return FLINT_MOE_ERR_INVALID_ARG;
  return flint_moe_enable_kernel_timing(st->h, enable);
}

flint_moe_status flint_moe_stack_read_trace(flint_moe_stack_t st, unsigned long long* out, int cap, int* n) {
  if (!st) return FLINT_MOE_ERR_INVALID_ARG;
  return flint_moe_read_trace(st->h, out, cap, n);
}

flint_moe_status flint_moe_stack_destroy(flint_moe_stack_t st) {
  if (!st) return FLINT_MOE_ERR_INVALID_ARG;
  flint_moe_destroy(st->h);
  delete st;
  return FLINT_MOE_OK;
}

}  // extern "C"

// ------------------------------------------------------------------------------------------
// Allocation-free forward.
//
// Some callers cannot allocate device memory at the point where they run the layer: a host
// application that owns every byte of device memory and hands plugins no allocator, a runtime
// that plans all of its memory at start-up and forbids allocation afterwards, or a latency
// path that cannot afford the implicit synchronisation of cudaMalloc.  For them this entry
// point takes its scratch space from one fixed array in device memory that the library
// declares itself, so the caller supplies only the weights, the input and the output.
//
// The array (25 MiB) holds the workspace of a handle with max_tokens = NOALLOC_MAX_T.
// Every GPU that loads the library reserves it until the process exits.  All calls on a
// device share it: calls whose work overlaps on the GPU (on different streams, or from
// different threads) race on it and must be serialised by the caller.  The barrier counters
// and tickets, which must start at zero, are cleared on the caller's stream at the start of
// every call; the status word is not: a device error (a bounded wait that ran out, an index
// out of range) stays recorded until flint_moe_noalloc_poll_device_status reads and clears it.
//
// The array's device address is looked up once per device and kept for the life of the
// process.  It belongs to the device's primary context: after cudaDeviceReset (or anything
// else that destroys and recreates that context) the kept address is stale, so these entry
// points must not be used on that device again in the same process.
namespace {

constexpr int NOALLOC_MAX_T = 4;
constexpr size_t NOALLOC_BYTES = size_t(25) << 20;
constexpr int NOALLOC_MAX_DEVICES = 64;

__device__ __align__(256) uint8_t g_noalloc_scratch[NOALLOC_BYTES];

std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[NOALLOC_MAX_DEVICES];
int g_noalloc_sms[NOALLOC_MAX_DEVICES];

// First call on a device (with that device current): the device address of the array, the
// kernel's shared-memory limit and occupancy, and a synchronous clear of the array's status
// word and counters.  Later calls reuse the address.
flint_moe_status noalloc_setup(int dev, void** ptr, int* n_sm) {
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return FLINT_MOE_ERR_CUDA;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
      return FLINT_MOE_ERR_CUDA;
    if (cudaFuncSetAttribute(decode_fused<MODE_MOE>, cudaFuncAttributeMaxDynamicSharedMemorySize, FUSED_SMEM) !=
        cudaSuccess)
      return FLINT_MOE_ERR_CUDA;
    // the cooperative launch needs one CTA resident on every SM (as flint_moe_create checks)
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_fused<MODE_MOE>, NTHREADS, FUSED_SMEM) !=
        cudaSuccess)
      return FLINT_MOE_ERR_CUDA;
    if (per_sm < 1) return FLINT_MOE_ERR_UNSUPPORTED;
    // the status word starts clear (later calls clear only the counters and tickets)
    if (cudaMemset(p, 0, make_layout(NOALLOC_MAX_T).zero_end) != cudaSuccess) return FLINT_MOE_ERR_CUDA;
    g_noalloc_sms[dev] = sms;
    g_noalloc_ptr[dev] = p;
  }
  *ptr = g_noalloc_ptr[dev];
  *n_sm = g_noalloc_sms[dev];
  return FLINT_MOE_OK;
}

}  // namespace

extern "C" flint_moe_status flint_moe_forward_noalloc(const flint_moe_weights* w, const void* x, int T, void* y,
                                                      int32_t* topk_idx, float* topk_w, flint_stream_t stream) {
  if (!w || !w->w_router || !w->w_gate || !w->w_up || !w->w_down || !w->ws_gate || !w->ws_up || !w->ws_down)
    return FLINT_MOE_ERR_INVALID_ARG;
  const void* ptrs[] = {w->w_router, w->w_gate, w->w_up, w->w_down, w->ws_gate, w->ws_up, w->ws_down, x, y};
  for (const void* q : ptrs)
    if (!q || !aligned16(q)) return FLINT_MOE_ERR_INVALID_ARG;
  if (w->router_bias && (reinterpret_cast<uintptr_t>(w->router_bias) & 3u)) return FLINT_MOE_ERR_INVALID_ARG;
  if (T < 1) return FLINT_MOE_ERR_INVALID_ARG;
  if (T > NOALLOC_MAX_T) return FLINT_MOE_ERR_UNSUPPORTED;  // beyond the fixed scratch array
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= NOALLOC_MAX_DEVICES) return FLINT_MOE_ERR_CUDA;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return FLINT_MOE_ERR_CUDA;
  if (major != 10 || minor != 3) return FLINT_MOE_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  int n_sm = 0;
  flint_moe_status s = noalloc_setup(dev, &scratch, &n_sm);
  if (s != FLINT_MOE_OK) return s;

  flint_moe_s h{};  // a handle on the stack: no host or device allocation
  h.cfg = flint_moe_config{H, E, K, I, IS, NOALLOC_MAX_T, 0u, 1e-6f};
  h.w = *w;
  h.sw = IS;
  h.dense = 0;
  h.device = dev;
  h.n_sm = n_sm;
  h.ws = static_cast<uint8_t*>(scratch);
  h.L = make_layout(NOALLOC_MAX_T);
  if (h.L.total > NOALLOC_BYTES) return FLINT_MOE_ERR_WORKSPACE;
  h.ws_bytes = NOALLOC_BYTES;
  h.timing = false;
  h.trace = false;
  h.n_ev = 0;
  const auto sw = CU_TENSOR_MAP_SWIZZLE_128B;
  const bool ok = make_map(&h.smaps.wr, w->w_router, H, E, 64, RT_ROWS, sw) &&
                  make_map(&h.smaps.wg, w->w_gate, (uint64_t)E * H, I, 64, GU_ROWS, sw) &&
                  make_map(&h.smaps.wu, w->w_up, (uint64_t)E * H, I, 64, GU_ROWS, sw) &&
                  make_map(&h.smaps.wd, w->w_down, (uint64_t)E * I, H, 64, DN_ROWS, sw) &&
                  make_map(&h.smaps.wsg, w->ws_gate, H, IS, 64, GU_ROWS, sw) &&
                  make_map(&h.smaps.wsu, w->ws_up, H, IS, 64, GU_ROWS, sw) &&
                  make_map(&h.smaps.wsd, w->ws_down, IS, H, 64, DN_ROWS, sw);
  if (!ok) return FLINT_MOE_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // barrier counters and tickets start at zero on every call; the status word (and the word
  // after it, which the timeout test waits on) is left for flint_moe_noalloc_poll_device_status
  if (cudaMemsetAsync(h.ws + h.L.bar_count, 0, h.L.zero_end - h.L.bar_count, st) != cudaSuccess)
    return FLINT_MOE_ERR_CUDA;
  Params p = make_params(&h, x, T, y, topk_idx, topk_w, nullptr);
  return run_decode(&h, p, st, true);
}

extern "C" flint_moe_status flint_moe_noalloc_poll_device_status(flint_stream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= NOALLOC_MAX_DEVICES) return FLINT_MOE_ERR_CUDA;
  void* scratch = nullptr;
  int n_sm = 0;
  flint_moe_status s = noalloc_setup(dev, &scratch, &n_sm);
  if (s != FLINT_MOE_OK) return s;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return FLINT_MOE_ERR_CUDA;
  const Layout L = make_layout(NOALLOC_MAX_T);
  uint8_t* ws = static_cast<uint8_t*>(scratch);
  uint32_t word = 0;
  if (cudaMemcpy(&word, ws + L.status, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess) return FLINT_MOE_ERR_CUDA;
  if (word == 0) return FLINT_MOE_OK;
  // a device error may leave tickets mid-count: clear them with the status word
  if (cudaMemset(ws + L.status, 0, L.zero_end - L.status) != cudaSuccess) return FLINT_MOE_ERR_CUDA;
  return (word & ST_TIMEOUT) ? FLINT_MOE_ERR_DEVICE_TIMEOUT : FLINT_MOE_ERR_DEVICE_BOUNDS;
}

// ------------------------------------------------------------------------------------------
// The dense SwiGLU MLP layers (serving-kit post, "The architecture, from the config": the
// model's first two layers are dense MLP layers, mlp_only_layers [0, 1], about 75M parameters
// for the two, i.e. width 6144).  A dense layer is run as the MoE layer's shared-expert path
// alone, at width ID: the decode-size kernel's shared gate/up and down steps up to 256 tokens,
// the tensor-core path's shared gate/up and down tiles above.
struct flint_dense_s {
  flint_moe_t h;
};

namespace {

flint_moe_status check_dense_config(const flint_dense_config* c) {
  if (!c) return FLINT_MOE_ERR_INVALID_ARG;
  if (c->hidden != H || c->inter != ID) return FLINT_MOE_ERR_UNSUPPORTED;
  if (c->max_tokens < 1 || c->max_tokens > MAX_TOKENS_LIMIT) return FLINT_MOE_ERR_INVALID_ARG;
  if (c->flags & ~(FLINT_MOE_FLAG_PRE_RMSNORM | FLINT_MOE_FLAG_RESIDUAL | FLINT_MOE_FLAG_TEST_WAIT_TIMEOUT))
    return FLINT_MOE_ERR_UNSUPPORTED;
  if ((c->flags & FLINT_MOE_FLAG_PRE_RMSNORM) && !(c->rms_eps > 0.f)) return FLINT_MOE_ERR_INVALID_ARG;
  return FLINT_MOE_OK;
}

flint_moe_config moe_config_of(const flint_dense_config* c) {
  return flint_moe_config{H, E, K, I, IS, c->max_tokens, c->flags, c->rms_eps};
}

}  // namespace

extern "C" {

flint_moe_status flint_dense_workspace_bytes(const flint_dense_config* cfg, size_t* bytes) {
  const flint_moe_status s = check_dense_config(cfg);
  if (s != FLINT_MOE_OK) return s;
  if (!bytes) return FLINT_MOE_ERR_INVALID_ARG;
  *bytes = make_layout(cfg->max_tokens, ID, true).total;
  return FLINT_MOE_OK;
}

flint_moe_status flint_dense_create(const flint_dense_config* cfg, const flint_dense_weights* w, void* workspace,
                                    size_t workspace_bytes, flint_dense_t* out) {
  if (!out) return FLINT_MOE_ERR_INVALID_ARG;
  *out = nullptr;
  flint_moe_status s = check_dense_config(cfg);
  if (s != FLINT_MOE_OK) return s;
  if (!w || !w->w_gate || !w->w_up || !w->w_down) return FLINT_MOE_ERR_INVALID_ARG;
  if (!aligned16(w->w_gate) || !aligned16(w->w_up) || !aligned16(w->w_down)) return FLINT_MOE_ERR_INVALID_ARG;
  flint_moe_weights mw{};
  mw.ws_gate = w->w_gate;
  mw.ws_up = w->w_up;
  mw.ws_down = w->w_down;
  const flint_moe_config mc = moe_config_of(cfg);
  flint_dense_s* d = new (std::nothrow) flint_dense_s();
  if (!d) return FLINT_MOE_ERR_CUDA;
  s = create_handle(&mc, &mw, workspace, workspace_bytes, ID, true, &d->h);
  if (s != FLINT_MOE_OK) {
    delete d;
    return s;
  }
  *out = d;
  return FLINT_MOE_OK;
}

flint_moe_status flint_dense_forward(flint_dense_t d, const void* x, int T, void* y, flint_stream_t stream) {
  if (!d) return FLINT_MOE_ERR_INVALID_ARG;
  return flint_moe_forward(d->h, x, T, y, nullptr, nullptr, stream);
}

flint_moe_status flint_dense_poll_device_status(flint_dense_t d, flint_stream_t stream) {
  if (!d) return FLINT_MOE_ERR_INVALID_ARG;
  return flint_moe_poll_device_status(d->h, stream);
}

flint_moe_status flint_dense_enable_kernel_timing(flint_dense_t d, int enable) {
  if (!d) return FLINT_MOE_ERR_INVALID_ARG;
  return flint_moe_enable_kernel_timing(d->h, enable);
}

flint_moe_status flint_dense_kernel_times(flint_dense_t d, const char** names, float* ms, int cap, int* n) {
  if (!d) return FLINT_MOE_ERR_INVALID_ARG;
  return flint_moe_kernel_times(d->h, names, ms, cap, n);
}

flint_moe_status flint_dense_destroy(flint_dense_t d) {
  if (!d) return FLINT_MOE_ERR_INVALID_ARG;
  flint_moe_destroy(d->h);
  delete d;
  return FLINT_MOE_OK;
}

}  // extern "C"

// ------------------------------------------------------------------------------------------
// Decode attention of the sliding-window layers (swa_attention.cuh).  The workspace: the status
// word, one ticket per (sequence, KV head), the chunk partials.
namespace {

constexpr int SWA_MAX_BATCH = 65535;  // the grid's z extent

struct SwaLayout {
  size_t status, ticket, zero_end, part, total;
};

SwaLayout swa_layout(int max_batch) {
  SwaLayout L{};
  L.status = 0;
  L.ticket = 256;
  L.zero_end = align_up(L.ticket + sizeof(uint32_t) * (size_t)max_batch * swa::NKV, 256);
  L.part = L.zero_end;
  L.total = align_up(L.part + sizeof(float) * (size_t)max_batch * swa::NH * swa::NSPLIT * swa::PSTRIDE, 256);
  return L;
}

// The largest batch a workspace of `bytes` holds (0 if none).
int swa_capacity(size_t bytes) {
  int lo = 0, hi = SWA_MAX_BATCH;
  while (lo < hi) {
    const int mid = (lo + hi + 1) / 2;
    if (swa_layout(mid).total <= bytes)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

}  // namespace

extern "C" {

flint_moe_status flint_swa_workspace_bytes(int max_batch, size_t* bytes) {
  if (!bytes || max_batch < 1 || max_batch > SWA_MAX_BATCH) return FLINT_MOE_ERR_INVALID_ARG;
  *bytes = swa_layout(max_batch).total;
  return FLINT_MOE_OK;
}

flint_moe_status flint_swa_workspace_init(void* workspace, size_t workspace_bytes, flint_stream_t stream) {
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return FLINT_MOE_ERR_WORKSPACE;
  const int cap = swa_capacity(workspace_bytes);
  if (cap < 1) return FLINT_MOE_ERR_WORKSPACE;
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return FLINT_MOE_ERR_CUDA;
  if (major != 10 || minor != 3) return FLINT_MOE_ERR_UNSUPPORTED;
  const SwaLayout L = swa_layout(cap);
  if (cudaFuncSetAttribute(swa::decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, swa::SMEM_BYTES) !=
      cudaSuccess)
    return FLINT_MOE_ERR_CUDA;
  return cudaMemsetAsync(workspace, 0, L.zero_end, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? FLINT_MOE_OK
             : FLINT_MOE_ERR_CUDA;
}

flint_moe_status flint_swa_decode(void* workspace, size_t workspace_bytes, const void* q, const void* k_cache,
                                  const void* v_cache, const float* sinks, const int32_t* pos, int B, void* out,
                                  flint_stream_t stream) {
  if (!q || !k_cache || !v_cache || !sinks || !pos || !out) return FLINT_MOE_ERR_INVALID_ARG;
  const void* ptrs[] = {q, k_cache, v_cache, out};
  for (const void* x : ptrs)
    if (!aligned16(x)) return FLINT_MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(sinks) & 3u) || (reinterpret_cast<uintptr_t>(pos) & 3u))
    return FLINT_MOE_ERR_INVALID_ARG;
  if (B < 1 || B > SWA_MAX_BATCH) return FLINT_MOE_ERR_INVALID_ARG;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return FLINT_MOE_ERR_WORKSPACE;
  const int cap = swa_capacity(workspace_bytes);
  if (B > cap) return FLINT_MOE_ERR_WORKSPACE;
  const SwaLayout L = swa_layout(cap);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  swa::Params p{};
  p.q = static_cast<const bf16*>(q);
  p.k = static_cast<const bf16*>(k_cache);
  p.v = static_cast<const bf16*>(v_cache);
  p.sinks = sinks;
  p.pos = pos;
  p.out = static_cast<bf16*>(out);
  p.B = B;
  p.part = reinterpret_cast<float*>(ws + L.part);
  p.ticket = reinterpret_cast<uint32_t*>(ws + L.ticket);
  p.status = reinterpret_cast<uint32_t*>(ws + L.status);
  // one CTA per (sequence, KV head) walking the 9 chunks once the batch has a pair per SM; below,
  // each pair split over 9 CTAs of one chunk (merged by the last of them)
  int dev = 0, n_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess)
    return FLINT_MOE_ERR_CUDA;
  const int nsplit = B * swa::NKV >= n_sm ? 1 : swa::NSPLIT;
  swa::decode_kernel<<<dim3(nsplit, swa::NKV, B), swa::NT, swa::SMEM_BYTES, reinterpret_cast<cudaStream_t>(stream)>>>(
      p);
  return cudaGetLastError() == cudaSuccess ? FLINT_MOE_OK : FLINT_MOE_ERR_CUDA;
}

flint_moe_status flint_swa_poll_device_status(void* workspace, flint_stream_t stream) {
  if (!workspace) return FLINT_MOE_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return FLINT_MOE_ERR_CUDA;
  uint32_t word = 0;
  if (cudaMemcpy(&word, workspace, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess) return FLINT_MOE_ERR_CUDA;
  if (word == 0) return FLINT_MOE_OK;
  if (cudaMemset(workspace, 0, sizeof word) != cudaSuccess) return FLINT_MOE_ERR_CUDA;
  return (word & ST_TIMEOUT) ? FLINT_MOE_ERR_DEVICE_TIMEOUT : FLINT_MOE_ERR_DEVICE_BOUNDS;
}

}  // extern "C"

// ------------------------------------------------------------------------------------------
// NVFP4 expert weights (decode sizes): the handle carries the codes, scales and tensor scales of
// the routed and shared experts; the router stays bf16.  Every call runs the decode-size kernel
// with its NVFP4 stream (decode_fused.cuh).
extern "C" flint_moe_status flint_moe_create_nvfp4(const flint_moe_config* cfg, const flint_moe_nvfp4_weights* w,
                                                   void* workspace, size_t workspace_bytes, flint_moe_t* out) {
  if (!out) return FLINT_MOE_ERR_INVALID_ARG;
  *out = nullptr;
  flint_moe_status s = check_config(cfg);
  if (s != FLINT_MOE_OK) return s;
  if (cfg->max_tokens > FP4_MAX_T) return FLINT_MOE_ERR_UNSUPPORTED;
  if (!w || !w->w_router || !aligned16(w->w_router)) return FLINT_MOE_ERR_INVALID_ARG;
  const void* ptrs[] = {w->gate_codes, w->up_codes, w->down_codes, w->gate_scales, w->up_scales, w->down_scales,
                        w->sgate_codes, w->sup_codes, w->sdown_codes, w->sgate_scales, w->sup_scales, w->sdown_scales};
  for (const void* q : ptrs)
    if (!q || !aligned16(q)) return FLINT_MOE_ERR_INVALID_ARG;
  if (!w->gate_tscale || !w->up_tscale || !w->down_tscale) return FLINT_MOE_ERR_INVALID_ARG;
  if (w->router_bias && (reinterpret_cast<uintptr_t>(w->router_bias) & 3u)) return FLINT_MOE_ERR_INVALID_ARG;
  // the handle's bf16 maps cover the router only; the expert maps are the NVFP4 ones
  flint_moe_weights bw{};
  bw.w_router = w->w_router;
  bw.router_bias = w->router_bias;
  s = create_handle(cfg, &bw, workspace, workspace_bytes, IS, false, out, true);
  if (s != FLINT_MOE_OK) return s;
  flint_moe_t h = *out;
  h->fp4 = 1;
  h->q = *w;
  Fp4Maps m;
  const uint64_t EH = (uint64_t)E * H, EI = (uint64_t)E * I;
  const bool ok =
      make_map_fp4_rows(&m.qg, w->gate_codes, EI) && make_map_fp4_rows(&m.qu, w->up_codes, EI) &&
      make_map_fp4_rows(&m.qsg, w->sgate_codes, IS) && make_map_fp4_rows(&m.qsu, w->sup_codes, IS) &&
      make_map_u8(&m.qd, w->down_codes, EH, I / 2, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B) &&
      make_map_u8(&m.qsd, w->sdown_codes, H, IS / 2, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B) &&
      make_map_u8(&m.sg, w->gate_scales, EI, H / 16, 128, FP4_GU_COLS) &&
      make_map_u8(&m.su, w->up_scales, EI, H / 16, 128, FP4_GU_COLS) &&
      make_map_u8(&m.ssg, w->sgate_scales, IS, H / 16, 128, FP4_GU_COLS) &&
      make_map_u8(&m.ssu, w->sup_scales, IS, H / 16, 128, FP4_GU_COLS) &&
      make_map_u8(&m.sd, w->down_scales, EH / 4, 128, 128, 32) &&  // [E*H][32 B] viewed as [E*H/4][128 B]
      make_map_u8(&m.ssd, w->sdown_scales, H, IS / 16, FP4_DN_ROWS / 16, 128) &&
      cudaMemcpy(h->ws + h->L.fp4maps, &m, sizeof m, cudaMemcpyHostToDevice) == cudaSuccess;
  if (!ok) {
    flint_moe_destroy(h);
    *out = nullptr;
    return FLINT_MOE_ERR_CUDA;
  }
  return FLINT_MOE_OK;
}
