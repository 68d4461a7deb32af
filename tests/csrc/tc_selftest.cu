// Test infrastructure: a dense bf16 GEMM D = A B (A [M][K] row-major, B [K][N] row-major,
// D fp32) run on the library's tensor-core engine in either tile orientation (rows of A on
// the TMEM lanes, or columns of B on the lanes with the rows of A as the MMA's N), so that its
// descriptors, TMA boxes, MMA pipeline and TMEM epilogue can be checked against torch.matmul.
// Not part of the product.
#include <cudaTypedefs.h>

#include "../../sparse_moe_layer_15_b300/csrc/tc_gemm.cuh"

using namespace flint;
using namespace flint::tc;

template <bool kCols>
struct TestGemm {
  static constexpr bool kColumns = kCols;
  CUtensorMap a, b;
  float* D;
  int M, N, K;
  int rpt;         // COLUMNS: rows per tile (16..256, multiple of 16)
  int skip_store;  // 1: the epilogue reads TMEM but stores nothing (engine timing only)
  uint32_t* st;
  // ROWS tiles: 128 rows x 256 columns; COLUMNS tiles: 128 columns x rpt rows
  __device__ int row_tile() const { return kCols ? rpt : TM; }
  __device__ int col_tile() const { return kCols ? 128 : TN; }
  __device__ void prologue(uint8_t*) const {}
  __device__ int num_tiles(const uint8_t*) const { return ((M + row_tile() - 1) / row_tile()) * (N / col_tile()); }
  __device__ int kblocks() const { return K / TK; }
  __device__ uint32_t* status() const { return st; }
  __device__ unsigned long long* trace() const { return nullptr; }
  __device__ void tile(int i, TileInfo& t, const uint8_t*) const {
    const int nt = N / col_tile();
    const int mt = i / nt, ntile = i % nt;
    t.amap = &a;
    t.a_row0 = mt * row_tile();
    t.b_row0 = 0;
    for (int c = 0; c < 4; ++c) {
      t.bmap[c] = &b;
      t.bcol[c] = ntile * col_tile() + c * 64;
    }
    t.row0 = mt * row_tile();
    t.valid = min(row_tile(), M - mt * row_tile());
    t.col0 = ntile * col_tile();
    t.aux = 0;
    t.n = (t.valid + 15) & ~15;
  }
  __device__ void epilogue(const TileInfo& t, uint32_t trow, int row, uint8_t*, const uint8_t*) const {
    if constexpr (kCols) {
      // lane `row` = output column col0 + row; TMEM columns = rows row0 ..
#pragma unroll 1
      for (int c = 0; c * 32 < t.valid; ++c) {
        float v[32];
        tmem_ld32(trow + uint32_t(c * 32), v);
        if (skip_store) {
          if (v[0] == 12345.f) D[0] = v[31];  // keeps the TMEM load alive
          continue;
        }
#pragma unroll
        for (int q = 0; q < 32; ++q)
          if (c * 32 + q < t.valid) D[(size_t)(t.row0 + c * 32 + q) * N + t.col0 + row] = v[q];
      }
    } else {
#pragma unroll 1
    for (int c = 0; c < TN / 32; ++c) {
      float v[32];
      tmem_ld32(trow + uint32_t(c * 32), v);
      if (skip_store) {
        if (v[0] == 12345.f) D[0] = v[31];
        continue;
      }
      if (row < t.valid) {
        float4* dst = reinterpret_cast<float4*>(D + (size_t)(t.row0 + row) * N + t.col0 + c * 32);
#pragma unroll
        for (int q = 0; q < 8; ++q) dst[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
      }
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

template <bool kCols>
static int run(const void* A, const void* B, float* D, int M, int N, int K, int rows_per_tile, int skip_store,
               uint32_t* status, cudaStream_t stream) {
  TestGemm<kCols> g{};
  if (!encode(&g.a, A, M, K, 64, kCols ? XC_ROWS : TM) || !encode(&g.b, B, K, N, 64, TK)) return -1;
  g.D = D;
  g.M = M;
  g.N = N;
  g.K = K;
  g.rpt = rows_per_tile;
  g.skip_store = skip_store;
  g.st = status;
  cudaError_t e =
      cudaFuncSetAttribute(gemm_kernel<TestGemm<kCols>>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return int(e);
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int tiles = kCols ? ((M + rows_per_tile - 1) / rows_per_tile) * (N / 128) : ((M + TM - 1) / TM) * (N / TN);
  const int grid = tiles < sms ? tiles : sms;
  gemm_kernel<TestGemm<kCols>><<<grid, NUM_THREADS, SMEM_BYTES, stream>>>(g);
  return int(cudaGetLastError());
}

// mode 0: ROWS tiles, 1: COLUMNS tiles of rows_per_tile rows (16..256, a multiple of 16);
// skip_store: time the engine alone.  Returns 0 on success, -1 on bad arguments, a CUDA error
// code otherwise.
extern "C" int tc_selftest_gemm_ex(const void* A, const void* B, float* D, int M, int N, int K, int mode,
                                   int rows_per_tile, int skip_store, uint32_t* status, void* stream) {
  if (M < 1 || N % TN || K % TK || !A || !B || !D || !status) return -1;
  if (mode != 0 && mode != 1) return -1;
  if (mode == 1 && (rows_per_tile < 16 || rows_per_tile > 256 || rows_per_tile % 16)) return -1;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return mode ? run<true>(A, B, D, M, N, K, rows_per_tile, skip_store, status, st)
              : run<false>(A, B, D, M, N, K, rows_per_tile, skip_store, status, st);
}

extern "C" int tc_selftest_gemm(const void* A, const void* B, float* D, int M, int N, int K, int mode,
                                uint32_t* status, void* stream) {
  return tc_selftest_gemm_ex(A, B, D, M, N, K, mode, 2 * TM, 0, status, stream);
}
