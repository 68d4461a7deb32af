// Tensor-core GEMM engine for sm_103a: tcgen05.mma with accumulators in TMEM, operands staged
// in shared memory by TMA, one persistent CTA per SM.
//
// Two operands:
//   X: activation rows, K-major (rows contiguous in K), TMA boxes of 64 (K) x 128 rows (ROWS)
//      or 64 (K) x 64 rows (COLUMNS), 128-byte swizzle;
//   W: weight columns, N-major (rows of W are contiguous in N, i.e. the matrices in y = x W
//      order), TMA boxes of 64 (N) x 64 (K rows), 128-byte swizzle, 8 KB each -- every box may
//      come from its own tensor map and column, so a tile can pair two matrices (gate | up).
// A launch runs all its tiles in one of two orientations (Problem::kColumns):
//   ROWS:    D[128 rows][256 cols] = X W, one MMA per K step (A = X, M = 128 rows; B = W,
//            N = 256 columns); TMEM lane = activation row, TMEM column = output column.
//            Pipeline: 4 stages of 48 KB (1 X box + 4 W boxes) per K block of 64.
//   COLUMNS: D[128 cols][n rows] = (X W)^T, one MMA per K step (A = W read N-major, M = 128
//            columns = W boxes 0 and 1; B = X read K-major, N = n rows, a multiple of 16 up to
//            256); TMEM lane = W column (box 0 on lanes 0..63, box 1 on 64..127), TMEM column =
//            activation row.  A group of rows costs its own size rounded up to 16 instead of
//            whole 128-row tiles.  Pipeline: 4 stages of [X: up to 4 boxes of 64 rows, only
//            ceil(n / 64) loaded, 32 KB | W: 2 boxes, 16 KB] per K block of 64.
//   Both read 12 KB of shared memory per 128 x 256 x 16 MMA.  Either way a tile owns 256 fp32
//   TMEM columns; two buffers, so the epilogue of one tile overlaps the main loop of the next.
// Warp roles: warp 0 issues TMA (one lane), warp 1 allocates TMEM and issues the MMAs (one
// lane), warps 2-5 run the epilogue (warp w reads TMEM lanes 32*(w%4) .. +31, one row each).
// Every wait is bounded (1 s); on expiry the device status word gets ST_TIMEOUT and the CTA
// aborts: a shared abort flag stops every role from issuing more work, the producer waits
// (bounded) for the TMA loads it has issued to land, the MMA issuer commits and waits
// (bounded) for the MMAs it has issued, and only then is TMEM released and the CTA ends, so
// no asynchronous copy or MMA is left in flight on freed shared memory or TMEM.
//
// A Problem class supplies the tile list and the epilogue:
//   static constexpr bool kColumns;            // orientation of every tile
//   void prologue(uint8_t* tbl) const;          // all threads, once: fill the table region
//   int num_tiles(const uint8_t* tbl) const;
//   int kblocks() const;                        // K blocks of 64 per tile, unless TileInfo::nkb says otherwise
//   void tile(int i, TileInfo& t, const uint8_t* tbl) const;  // operand maps and coordinates
//   void epilogue(const TileInfo& t, uint32_t tmem_row, int row, uint8_t* epi,
//                 const uint8_t* tbl) const;
//        called by each epilogue thread for its TMEM lane `row` (0..127: a tile row in ROWS
//        mode, an output column in COLUMNS mode); tmem_row addresses column 0 of that lane's
//        accumulator (load with tmem_ld32, warp-collective, so every lane loads before any
//        lane branches on its row); epi_sync() synchronises the 128 epilogue threads
//   uint32_t* status() const;
//   unsigned long long* trace() const;  // null, or 8 slots of a TRACE_SLOTS-wide row per CTA
//        that receive the CTA's wait profile: SM cycles the producer waited for free slots,
//        the MMA issuer for loaded slots and for free accumulators, the first epilogue warp
//        for full accumulators and inside the epilogue; the global timer (ns) at the start and
//        the end; the tiles processed.
#pragma once

#include "common.cuh"

namespace flint {
namespace tc {

constexpr int TM = 128;
constexpr int TN = 256;
constexpr int TK = 64;
constexpr int KSTEP = 16;
constexpr int STAGES = 4;
constexpr int A_BYTES = TM * TK * 2;            // 16 KB
constexpr int XC_ROWS = 64;                     // rows of a COLUMNS-mode X box
constexpr int XC_BYTES = XC_ROWS * TK * 2;      // 8 KB
constexpr int B_CHUNK = TK * 64 * 2;            // 8 KB: 64 K rows x 64 columns
constexpr int B_BYTES = 4 * B_CHUNK;            // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;  // 48 KB
constexpr int NUM_THREADS = 192;
constexpr uint32_t TMEM_COLS = 512;
constexpr int EPI_SMEM = 8192;  // per-CTA scratch handed to the epilogue
constexpr int align_up_c(int v, int a) { return (v + a - 1) / a * a; }
constexpr int TBL_SMEM = 4096;  // per-CTA table filled by the problem's prologue

// kind::f16 instruction descriptors: D fp32 (bits 4-5 = 1), A and B bf16 (bits 7-9 and
// 10-12 = 1), bit 15 = A MN-major, bit 16 = B MN-major, N >> 3 at bit 17, M >> 4 at bit 24.
// ROWS: A = X K-major, B = W N-major, N = 256, M = 128.
constexpr uint32_t IDESC = (1u << 4) | (1u << 7) | (1u << 10) | (0u << 15) | (1u << 16) |
                           (uint32_t(TN >> 3) << 17) | (uint32_t(TM >> 4) << 24);
// COLUMNS: A = W N-major (M = 128 of its columns), B = X K-major (N = n rows, <= 256).
__host__ __device__ constexpr uint32_t idesc_columns(int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (1u << 15) | (0u << 16) | (uint32_t(n >> 3) << 17) |
         (uint32_t(TM >> 4) << 24);
}

struct Smem {
  static constexpr int stages = 0;  // STAGES x 48 KB
  static constexpr int bars = stages + STAGES * STAGE_BYTES;  // 16 mbarriers
  static constexpr int tmem_slot = bars + 8 * 16;
  static constexpr int epi = align_up_c(tmem_slot + 16, 128);
  static constexpr int tbl = epi + EPI_SMEM;
  static constexpr int bytes = tbl + TBL_SMEM;
};
constexpr int SMEM_BYTES = Smem::bytes + 1024;
constexpr int BAR_FULL = 0, BAR_EMPTY = 4, BAR_TFULL = 8, BAR_TEMPTY = 10, BAR_DRAIN = 12;
// tmem_slot[0]: the TMEM base address written by tcgen05.alloc; tmem_slot[1]: the abort flag.

struct TileInfo {
  const CUtensorMap* amap;  // X operand (activation rows)
  int a_row0;               // first X row (TMA coordinate)
  int b_row0;               // first W row (K offset of the weight matrix in its tensor map)
  const CUtensorMap* bmap[4];
  int bcol[4];              // column (N) coordinate of each of the four W boxes
  int row0;                 // problem-specific: first output row
  int valid;                // rows of this tile that are real
  int col0;                 // problem-specific: first output column
  int aux;                  // problem-specific
  int n = 0;                // COLUMNS: rows fed to the MMA (valid rounded up to 16, <= 256)
  int nkb = 0;              // K blocks of this tile (0: Problem::kblocks())
};

// ------------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return uint64_t((saddr >> 4) & 0x3FFFu) | (uint64_t((lbo >> 4) & 0x3FFFu) << 16) |
         (uint64_t((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive fp32 columns of this thread's TMEM lane (warp-collective).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Bounded mbarrier wait that also gives up as soon as another role of the CTA has aborted
// (*abort != 0).  On expiry it records ST_TIMEOUT and raises the abort flag.  Returns false
// when the phase did not complete.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, uint32_t* status,
                                         volatile uint32_t* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (*abort) return false;
    if (globaltimer_ns() - t0 > WAIT_LIMIT_NS) {
      record_status(status, ST_TIMEOUT);
      *abort = 1u;
      return false;
    }
  }
  return true;
}

// Drain wait after an abort: bounded by the wait limit only (the abort flag is already up).
__device__ __forceinline__ void drain_bar(uint64_t* bar, uint32_t parity, uint32_t* status) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > WAIT_LIMIT_NS) {
      record_status(status, ST_TIMEOUT);
      return;
    }
  }
}

// Barrier among the four epilogue warps (128 threads).
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 2, 128;" ::: "memory"); }

// Barrier among the four epilogue warps that also returns true in every one of them when `fail`
// is true in any: they skip a tile (and end) together, never some of them entering the
// epilogue's own barriers without the others.
__device__ __forceinline__ bool epi_any(bool fail) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\t"
      "bar.red.or.pred p, 2, 128, q;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"(fail ? 1u : 0u)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ uint8_t* align1024(uint8_t* raw) {
  const uint32_t a = smem_u32(raw);
  return raw + ((1024u - (a & 1023u)) & 1023u);
}

// ------------------------------------------------------------------ the kernel
template <class Problem>
__global__ void __launch_bounds__(NUM_THREADS, 1) gemm_kernel(const __grid_constant__ Problem prob) {
  constexpr bool cols = Problem::kColumns;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + Smem::bars);
  uint64_t* tfull = bars + BAR_TFULL;
  uint64_t* tempty = bars + BAR_TEMPTY;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + Smem::tmem_slot);
  volatile uint32_t* abort = tmem_slot + 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint32_t* status = prob.status();
  unsigned long long* trace = prob.trace();
  if (trace) trace += (size_t)blockIdx.x * TRACE_SLOTS;
  if (trace && threadIdx.x == 0) trace[5] = globaltimer_ns();

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bars + BAR_FULL + s, 1);
      mbar_init(bars + BAR_EMPTY + s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull + b, 1);
      mbar_init(tempty + b, 4);  // one arrival per epilogue warp
    }
    mbar_init(bars + BAR_DRAIN, 1);
    *abort = 0u;
    fence_mbar_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  pdl_launch_dependents();
  pdl_wait();
  uint8_t* tbl = sm + Smem::tbl;
  prob.prologue(tbl);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int ntiles = prob.num_tiles(tbl);
  const int kb_n = prob.kblocks();

  if (warp == 0) {
    // ---------------- producer
    long long w_wait = 0;
    int pos = 0;  // stages issued
    if constexpr (cols) {
      if (lane == 0) {
        for (int i = blockIdx.x; i < ntiles && !*abort; i += gridDim.x) {
          TileInfo t;
          prob.tile(i, t, tbl);
          const int nxb = (t.n + XC_ROWS - 1) / XC_ROWS;  // 1..4 X boxes of 64 rows
          const int nkb = t.nkb ? t.nkb : kb_n;
          for (int kb = 0; kb < nkb; ++kb, ++pos) {
            const int st = pos % STAGES, use = pos / STAGES;
            const long long c0 = clock64();
            if (use > 0 && !wait_bar(bars + BAR_EMPTY + st, uint32_t(use - 1) & 1u, status, abort)) break;
            if (*abort) break;
            w_wait += clock64() - c0;
            uint8_t* x = sm + Smem::stages + st * STAGE_BYTES;
            uint8_t* w = x + 2 * A_BYTES;
            uint64_t* full = bars + BAR_FULL + st;
            mbar_arrive_expect_tx(full, uint32_t(nxb * XC_BYTES + 2 * B_CHUNK));
            for (int c = 0; c < nxb; ++c) tma_load_2d(x + c * XC_BYTES, t.amap, kb * TK, t.a_row0 + c * XC_ROWS, full);
            tma_load_2d(w, t.bmap[0], t.bcol[0], t.b_row0 + kb * TK, full);
            tma_load_2d(w + B_CHUNK, t.bmap[1], t.bcol[1], t.b_row0 + kb * TK, full);
          }
        }
      }
    } else if (lane == 0) {
      for (int i = blockIdx.x; i < ntiles && !*abort; i += gridDim.x) {
        TileInfo t;
        prob.tile(i, t, tbl);
        const int nkb = t.nkb ? t.nkb : kb_n;
        for (int kb = 0; kb < nkb; ++kb, ++pos) {
          const int st = pos % STAGES, use = pos / STAGES;
          const long long c0 = clock64();
          if (use > 0 && !wait_bar(bars + BAR_EMPTY + st, uint32_t(use - 1) & 1u, status, abort)) break;
          if (*abort) break;
          w_wait += clock64() - c0;
          uint8_t* a = sm + Smem::stages + st * STAGE_BYTES;
          uint8_t* b = a + A_BYTES;
          mbar_arrive_expect_tx(bars + BAR_FULL + st, STAGE_BYTES);
          tma_load_2d(a, t.amap, kb * TK, t.a_row0, bars + BAR_FULL + st);
#pragma unroll
          for (int c = 0; c < 4; ++c)
            tma_load_2d(b + c * B_CHUNK, t.bmap[c], t.bcol[c], t.b_row0 + kb * TK, bars + BAR_FULL + st);
        }
      }
    }
    // the loads already issued must land before the CTA may end, also after an abort (the last
    // use of each slot is the only phase of its full barrier that can still be pending; without
    // an abort the MMA issuer has waited for them all, and these waits return at once)
    if (lane == 0)
      for (int st = 0; st < STAGES && st < pos; ++st)
        drain_bar(bars + BAR_FULL + st, uint32_t((pos - 1 - st) / STAGES) & 1u, status);
    if (trace && lane == 0) trace[0] = (unsigned long long)w_wait;
  } else if (warp == 1) {
    // ---------------- MMA issuer
    if (lane == 0) {
      int pos = 0, it = 0;
      bool issued = false;
      long long w_full = 0, w_tempty = 0;
      for (int i = blockIdx.x; i < ntiles && !*abort; i += gridDim.x, ++it) {
        TileInfo t;
        prob.tile(i, t, tbl);
        const uint32_t idesc = cols ? idesc_columns(t.n) : IDESC;
        const int buf = it & 1, use = it >> 1;
        long long c0 = clock64();
        if (use > 0 && !wait_bar(tempty + buf, uint32_t(use - 1) & 1u, status, abort)) break;
        w_tempty += clock64() - c0;
        tc_fence_after();
        const uint32_t d = tmem_base + uint32_t(buf * TN);
        const int nkb = t.nkb ? t.nkb : kb_n;
        bool done = true;
        for (int kb = 0; kb < nkb; ++kb, ++pos) {
          uint32_t x, w;
          c0 = clock64();
          const int st = pos % STAGES;
          if (!wait_bar(bars + BAR_FULL + st, uint32_t(pos / STAGES) & 1u, status, abort)) {
            done = false;
            break;
          }
          issued = true;
          x = smem_u32(sm + Smem::stages + st * STAGE_BYTES);
          w = x + (cols ? 2 : 1) * A_BYTES;
          w_full += clock64() - c0;
          tc_fence_after();
#pragma unroll
          for (int s = 0; s < TK / KSTEP; ++s) {
            // X K-major: a K step is 32 bytes along the swizzled row (8-row groups 1 KB apart);
            // W N-major: a K step is 16 rows of 128 bytes, 64-column boxes 8 KB apart
            const uint64_t xd = smem_desc(x + s * (KSTEP * 2), 16, 1024);
            const uint64_t wd = smem_desc(w + s * (KSTEP * 128), B_CHUNK, 1024);
            const uint32_t acc = (kb | s) != 0 ? 1u : 0u;
            if constexpr (cols)
              mma_bf16(d, wd, xd, idesc, acc);
            else
              mma_bf16(d, xd, wd, idesc, acc);
          }
          // the slots are free once these MMAs have read them
          mma_commit(bars + BAR_EMPTY + st);
        }
        if (!done) break;
        mma_commit(tfull + buf);  // the accumulator is complete
      }
      // every MMA issued completes before TMEM is released, also after an abort (without one,
      // the epilogue has waited for the last accumulator already)
      if (issued) {
        mma_commit(bars + BAR_DRAIN);
        drain_bar(bars + BAR_DRAIN, 0u, status);
      }
      if (trace) {
        trace[1] = (unsigned long long)w_full;
        trace[2] = (unsigned long long)w_tempty;
      }
    }
  } else {
    // ---------------- epilogue (warps 2..5)
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    int it = 0;
    long long w_tfull = 0, busy = 0;
    for (int i = blockIdx.x; i < ntiles; i += gridDim.x, ++it) {
      const int buf = it & 1;
      const long long c0 = clock64();
      // every thread waits itself; the four warps skip the tile (and end) together on an abort
      const bool ok = wait_bar(tfull + buf, uint32_t(it >> 1) & 1u, status, abort);
      if (epi_any(!ok)) break;
      tc_fence_after();
      const long long c1 = clock64();
      TileInfo t;
      prob.tile(i, t, tbl);
      const uint32_t trow = tmem_base + (uint32_t(quarter * 32) << 16) + uint32_t(buf * TN);
      prob.epilogue(t, trow, row, sm + Smem::epi, tbl);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty + buf);
      w_tfull += c1 - c0;
      busy += clock64() - c1;
    }
    if (trace && warp == 2 && lane == 0) {
      trace[3] = (unsigned long long)w_tfull;
      trace[4] = (unsigned long long)busy;
      trace[7] = (unsigned long long)it;
    }
  }
  // wait for the last accumulators to be consumed, then release TMEM
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (trace && threadIdx.x == 0) trace[6] = globaltimer_ns();
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS) : "memory");
}

}  // namespace tc
}  // namespace flint
