// Test infrastructure: a dense bf16 GEMM D = A B (A [M][K] row-major, B [K][N] row-major,
// D fp32) run on the library's tensor-core engine, so that its descriptors, TMA boxes, MMA
// pipeline and TMEM epilogue can be checked against torch.matmul.  Not part of the product.
#include <cudaTypedefs.h>

#include "../../sparse_moe_layer_15_b300/csrc/tc_gemm.cuh"

using namespace flint;
using namespace flint::tc;

struct TestGemm {
  CUtensorMap a, b;
  float* D;
  int M, N, K;
  uint32_t* st;
  __device__ void prologue(uint8_t*) const {}
  __device__ int num_tiles(const uint8_t*) const { return ((M + TM - 1) / TM) * (N / TN); }
  __device__ int kblocks() const { return K / TK; }
  __device__ uint32_t* status() const { return st; }
  __device__ void tile(int i, TileInfo& t, const uint8_t*) const {
    const int nt = N / TN;
    const int mt = i / nt, ntile = i % nt;
    t.amap = &a;
    t.a_row0 = mt * TM;
    t.b_row0 = 0;
    for (int c = 0; c < 4; ++c) {
      t.bmap[c] = &b;
      t.bcol[c] = ntile * TN + c * 64;
    }
    t.row0 = mt * TM;
    t.valid = min(TM, M - mt * TM);
    t.col0 = ntile * TN;
    t.aux = 0;
  }
  __device__ void epilogue(const TileInfo& t, uint32_t trow, int row, uint8_t*, const uint8_t*) const {
#pragma unroll 1
    for (int c = 0; c < TN / 32; ++c) {
      float v[32];
      tmem_ld32(trow + uint32_t(c * 32), v);
      if (row < t.valid) {
        float4* dst = reinterpret_cast<float4*>(D + (size_t)(t.row0 + row) * N + t.col0 + c * 32);
#pragma unroll
        for (int q = 0; q < 8; ++q) dst[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
      }
    }
  }
};

static bool encode(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t bc, uint32_t br) {
  static PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
  if (!enc) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess)
      return false;
    enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {bc, br};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Returns 0 on success, -1 on bad arguments, a CUDA error code otherwise.
extern "C" int tc_selftest_gemm(const void* A, const void* B, float* D, int M, int N, int K, uint32_t* status,
                                void* stream) {
  if (M < 1 || N % TN || K % TK || !A || !B || !D || !status) return -1;
  TestGemm g{};
  if (!encode(&g.a, A, M, K, 64, TM) || !encode(&g.b, B, K, N, 64, TK)) return -1;
  g.D = D;
  g.M = M;
  g.N = N;
  g.K = K;
  g.st = status;
  cudaError_t e = cudaFuncSetAttribute(gemm_kernel<TestGemm>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return int(e);
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int tiles = ((M + TM - 1) / TM) * (N / TN);
  const int grid = tiles < sms ? tiles : sms;
  gemm_kernel<TestGemm><<<grid, NUM_THREADS, SMEM_BYTES, static_cast<cudaStream_t>(stream)>>>(g);
  return int(cudaGetLastError());
}
