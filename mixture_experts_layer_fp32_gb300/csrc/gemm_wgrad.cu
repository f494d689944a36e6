// Weight gradients of the grouped SwiGLU experts (the backward's wgrad GEMMs)
// on the 5th-generation tensor cores:
//   dW[e] (M x N, fp32) = X_e^T . Y_e
// with X_e, Y_e the rows [offsets[e], offsets[e+1]) of X [rows, M] and
// Y [rows, N] (bf16; Y's row stride ldy): dW2[e] = H_e^T dY_e,
// dW1[e] = X_e^T da_e, dW3[e] = X_e^T dg_e.  The reduction runs over the
// expert's rows, whose number is only known on the device.
//
// Design (one CTA per SM, persistent, the roles of the forward kernel):
//  * Tile = (expert, 128 rows of M, 256 columns of N); the accumulator is a
//    128 x 256 fp32 block in TMEM (two buffers).  Tiles are listed expert by
//    expert, the smaller output dimension fastest; an expert with no rows
//    gets a zero block.
//  * K runs over the expert's rows in blocks of 64.  Both operands are
//    MN-major in shared memory (X's M and Y's N contiguous): per stage two
//    64 (M) x 64 (rows) boxes of X and four 64 (N) x 64 (rows) boxes of Y,
//    128-byte swizzle, 48 KB, 4 stages.
//  * An expert's last block also fetches the next expert's rows.  The MMA
//    steps 16 rows at a time, so it issues only the steps that hold one of
//    the expert's rows, and a seventh warp clears the rest of the last such
//    step: it waits for the copies, zeroes those (at most 15) rows in every
//    box of both operands (a swizzled 128-byte row stays one row; rows past
//    the permuted rows may hold any bits, so B is cleared too), makes the
//    writes visible to the tensor core (fence.proxy.async) and releases the
//    stage on a second barrier, which the MMA thread waits on instead.  The TMA producer never
//    waits for a copy.  The zeroing warp consumes every stage (it waits for
//    each fill and arrives on the stage's empty barrier beside the MMA's
//    commit), so it can neither lap the producer nor be lapped by it and
//    every parity wait sees the phase it means.
//  * The epilogue warps move each 32-column slice of the fp32 accumulator
//    from TMEM to a swizzled 4 KB staging block and one lane stores it with
//    TMA (two blocks per warp, so the store of one overlaps the drain of the
//    next); the output is 4 bytes per element, which makes this store the
//    bound of the GEMM when experts have few rows.
//  * Every wait is bounded as in the forward kernel (error word, abort flag,
//    drain before TMEM is freed).
#include <stdlib.h>

#include "common.cuh"
#include "sm100_ptx.cuh"

namespace moe {
namespace {

constexpr int WM = 128, WN = 256, WK = 64;         // tile M, N; rows per stage
constexpr int W_BOX = 64 * WK * 2;                 // 64 (M or N) x 64 rows, bf16: 8 KB
constexpr int W_A_BYTES = 2 * W_BOX;
constexpr int W_STAGE = W_A_BYTES + 4 * W_BOX;     // 48 KB
constexpr int W_STAGES = 4;
constexpr int W_THREADS = 224;                     // TMA, MMA, 4 epilogue warps, tail zeroing
// Output staging: per epilogue warp two 32 x 32 fp32 blocks (4 KB each) in
// the TMA's 128-byte swizzle (16-byte chunk j of row r at chunk j ^ (r % 8)),
// stored by TMA while the warp drains the next 32 columns.
constexpr int W_STG_BYTES = 4096;
constexpr int W_EPI_BYTES = 4 * 2 * W_STG_BYTES;
constexpr int W_NUM_BARS = 3 * W_STAGES + 5;       // full, masked, empty, acc_full[2], acc_empty[2], drain
constexpr int W_SMEM = 1024 + W_STAGES * W_STAGE + W_EPI_BYTES + W_NUM_BARS * 8 + 16 +
                       (MOE_MAX_EXPERTS + 1) * 4 + MOE_MAX_EXPERTS;
static_assert(MOE_MAX_EXPERTS <= 256, "the expert order is kept in bytes");
static_assert(W_SMEM <= 227 * 1024, "shared memory budget");
// kind::f16, bf16 A and B, fp32 D, A and B MN-major (bits 15 and 16), N=256, M=128
constexpr uint32_t W_IDESC = ptx::idesc_bf16_f32(WM, WN, /*b_mn_major=*/true) | (1u << 15);
constexpr long long kWaitCycles = 4000000000LL;

struct WgradArgs {
  const int32_t* offsets;
  int E, M, N;
  int64_t max_rows;
  float* out;  // [E, M, N]
  int* err;
};

struct WCtl {
  uint64_t* bar;
  volatile int* abort_flag;
  int* err;
  __device__ uint32_t full(int s) const { return ptx::smem_u32(bar + s); }
  __device__ uint32_t masked(int s) const { return ptx::smem_u32(bar + W_STAGES + s); }
  __device__ uint32_t empty(int s) const { return ptx::smem_u32(bar + 2 * W_STAGES + s); }
  __device__ uint32_t acc_full(int b) const { return ptx::smem_u32(bar + 3 * W_STAGES + b); }
  __device__ uint32_t acc_empty(int b) const { return ptx::smem_u32(bar + 3 * W_STAGES + 2 + b); }
  __device__ uint32_t drain() const { return ptx::smem_u32(bar + 3 * W_STAGES + 4); }
  __device__ bool wait(uint32_t b, uint32_t parity, int site, bool honour_abort = true) const {
    bool timed_out;
    if (ptx::mbar_wait_bounded(b, parity, kWaitCycles, abort_flag, honour_abort, &timed_out))
      return true;
    if (timed_out) report_error(err, DEV_ERR_TIMEOUT, site);
    return false;
  }
};

// The j-th tile of worker p of P (a CTA, or an SM pair), -1 past its last.
// Balanced loads (`zig` false): tile p + j*P, experts in index order.
// Skewed loads (`zig`: the largest expert has more than 4x the mean rows):
// the experts are sorted by rows, most first (see decode_wtile), and the
// tiles are taken from both ends of that list: wave j gives worker p the
// position g = j*P + (p+j) mod P of the sequence front, back, front, back...
// (g even: tile g/2; g odd: tile total-1-g/2).  The front tiles are long and
// bound by the MMA, the back ones short and bound by their fp32 stores: each
// wave puts half the workers on each kind and every worker alternates, so
// stores and MMAs overlap across the GPU instead of all workers moving
// through the same expert together.  Each end keeps an expert's tiles
// together (L2 reuse of its rows); balanced loads keep one expert at a time.
__device__ __forceinline__ int sched_tile(int j, int p, int P, int total, bool zig) {
  if (!zig) {
    const int tile = p + j * P;
    return tile < total ? tile : -1;
  }
  const int g = j * P + (p + j) % P;
  if (g >= total) return -1;
  return (g & 1) ? total - 1 - (g >> 1) : (g >> 1);
}

// Tiles listed expert by expert; inside an expert the smaller of the two
// output dimensions varies fastest (n_fast = N < M), so the tiles in flight
// together cover all of the smaller operand's columns and a few stripes of
// the larger one: the expert's rows of both stay in L2 while they are used
// (the other order streams the larger operand once per stripe of the smaller).
__device__ __forceinline__ void decode_wtile(int tile, int MT, int NT, bool n_fast,
                                             const uint8_t* ord, int& e, int& m0, int& n0,
                                             int tile_m = WM) {
  const int s = tile / (MT * NT);
  e = ord[s];
  const int u = tile - s * MT * NT;
  int mt, nt;
  if (n_fast) {
    mt = u / NT;
    nt = u - mt * NT;
  } else {
    nt = u / MT;
    mt = u - nt * MT;
  }
  m0 = mt * tile_m;
  n0 = nt * WN;
}

__device__ __forceinline__ void st_shared_v4(uint32_t a, uint32_t x, uint32_t y, uint32_t z,
                                             uint32_t w) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(x), "r"(y), "r"(z), "r"(w)
               : "memory");
}

// One epilogue warp drains its 32 accumulator rows (TMEM lanes; output rows
// orow .. orow+31 of dW viewed as [E*M, N]) for columns [0, valid), to
// output columns n0 + c, 32 columns per TMA store.  Lane 0 issues the stores
// and owns their bulk groups; `ck` counts this warp's stores across tiles
// (staging block ck & 1, reused once the store two back has read it).
__device__ __forceinline__ void drain_to_tma(uint32_t tb, const CUtensorMap* tmO, int orow, int n0,
                                             int valid, bool zero, uint32_t stg, int lane,
                                             uint32_t& ck) {
#pragma unroll 1
  for (int c = 0; c < valid; c += 32) {
    uint32_t y[32];
    ptx::tmem_ld32(tb + c, y);
    ptx::tmem_wait_ld();
    const uint32_t buf = stg + (ck & 1u) * W_STG_BYTES;
    if (ck >= 2 && lane == 0) ptx::bulk_wait_group_read<1>();
    __syncwarp();
    const uint32_t row = buf + lane * 128;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t a = row + ((j ^ (lane & 7)) << 4);
      if (zero)
        st_shared_v4(a, 0u, 0u, 0u, 0u);
      else
        st_shared_v4(a, y[4 * j], y[4 * j + 1], y[4 * j + 2], y[4 * j + 3]);
    }
    ptx::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      ptx::tma_store_2d(tmO, n0 + c, orow, buf);
      ptx::bulk_commit_group();
    }
    ++ck;
  }
}

__global__ void __launch_bounds__(W_THREADS, 1)
    tc_wgrad_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmY,
                    const __grid_constant__ CUtensorMap tmO, WgradArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* stages = smem;
  const uint32_t epi = ptx::smem_u32(smem + W_STAGES * W_STAGE);  // 1 KB aligned
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + W_STAGES * W_STAGE + W_EPI_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + W_NUM_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* off = reinterpret_cast<int*>(tmem_slot + 4);
  uint8_t* ord = reinterpret_cast<uint8_t*>(off + MOE_MAX_EXPERTS + 1);
  int* zig_word = reinterpret_cast<int*>(tmem_slot + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = args.E;
  const int MT = args.M / WM, NT = (args.N + WN - 1) / WN;
  const int total = E * MT * NT;
  const bool n_fast = args.N < args.M;
  const WCtl ctl{bars, abort_flag, args.err};

  if (threadIdx.x == 0) {
    for (int s = 0; s < W_STAGES; ++s) {
      ptx::mbar_init(ctl.full(s), 1);
      ptx::mbar_init(ctl.masked(s), 1);
      ptx::mbar_init(ctl.empty(s), 2);  // MMA commit + zeroing warp
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(ctl.acc_full(b), 1);
      ptx::mbar_init(ctl.acc_empty(b), 4);
    }
    ptx::mbar_init(ctl.drain(), 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
    ptx::prefetch_tensormap(&tmX);
    ptx::prefetch_tensormap(&tmY);
    ptx::prefetch_tensormap(&tmO);
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), 512);
    ptx::tmem_relinquish();
  }
  // no offsets: one dense group over rows [0, max_rows) (E == 1)
  for (int e = threadIdx.x; e <= E; e += blockDim.x)
    off[e] = args.offsets ? args.offsets[e] : (e == 0 ? 0 : static_cast<int>(args.max_rows));
  __syncthreads();
  if (threadIdx.x == 0) {  // offsets must start at 0, never decrease, end within the buffers
    bool ok = off[0] == 0 && off[E] <= args.max_rows;
    for (int e = 0; e < E; ++e) ok = ok && off[e + 1] >= off[e];
    if (!ok) {
      for (int e = 0; e <= E; ++e) off[e] = 0;
      if (blockIdx.x == 0) report_error(args.err, DEV_ERR_INDEX, -1);
    }
    int most = 0;
    for (int e = 0; e < E; ++e) most = max(most, off[e + 1] - off[e]);
    *zig_word = static_cast<int64_t>(most) * E > 4LL * off[E];
  }
  __syncthreads();
  const bool zig = *zig_word != 0;
  // skewed loads: experts by rows, most first (equal counts: lower index
  // first); balanced: index order
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int n = off[e + 1] - off[e];
    int r = e;
    if (zig) {
      r = 0;
      for (int q = 0; q < E; ++q) {
        const int m = off[q + 1] - off[q];
        r += (m > n) || (m == n && q < e);
      }
    }
    ord[r] = static_cast<uint8_t>(e);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      int stage = 0;
      uint32_t phase = 0;
      uint32_t fill_parity = 0, filled = 0;
      bool alive = true;
      for (int j = 0, tile; alive && (tile = sched_tile(j, blockIdx.x, gridDim.x, total, zig)) >= 0; ++j) {
        int e, m0, n0;
        decode_wtile(tile, MT, NT, n_fast, ord, e, m0, n0);
        const int r0 = off[e], rows = off[e + 1] - off[e];
        const int KB = (rows + WK - 1) / WK;
        for (int kb = 0; kb < KB; ++kb) {
          if (!ctl.wait(ctl.empty(stage), phase ^ 1u, 11)) {
            alive = false;
            break;
          }
          const uint32_t a = ptx::smem_u32(stages + stage * W_STAGE);
          const uint32_t b = a + W_A_BYTES;
          const int row = r0 + kb * WK;
          const uint32_t fb = ctl.full(stage);
          ptx::mbar_arrive_expect_tx(fb, W_STAGE);
          ptx::tma_load_2d(a, &tmX, m0, row, fb);
          ptx::tma_load_2d(a + W_BOX, &tmX, m0 + 64, row, fb);
#pragma unroll
          for (int q = 0; q < 4; ++q) ptx::tma_load_2d(b + q * W_BOX, &tmY, n0 + 64 * q, row, fb);
          filled |= 1u << stage;
          fill_parity = (fill_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == W_STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (alive) {
        for (int i = 0; i < W_STAGES; ++i) {
          if (!ctl.wait(ctl.empty(stage), phase ^ 1u, 13, false)) break;
          if (++stage == W_STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      } else {
        for (int s = 0; s < W_STAGES; ++s)
          if (filled >> s & 1u) ctl.wait(ctl.full(s), fill_parity >> s & 1u, 14, false);
      }
    }
  } else if (warp == 6) {
    // ------------------------------------------------ tail zeroing (the whole warp)
    int stage = 0;
    uint32_t phase = 0;
    bool alive = true;
    for (int j = 0, tile; alive && (tile = sched_tile(j, blockIdx.x, gridDim.x, total, zig)) >= 0; ++j) {
      int e, m0, n0;
      decode_wtile(tile, MT, NT, n_fast, ord, e, m0, n0);
      const int rows = off[e + 1] - off[e];
      const int KB = (rows + WK - 1) / WK;
      for (int kb = 0; kb < KB; ++kb) {
        const int valid = min(WK, rows - kb * WK);
        if (!__all_sync(0xffffffffu, ctl.wait(ctl.full(stage), phase, 12))) {
          alive = false;
          break;
        }
        if (valid < WK) {
          // rows [valid, valid rounded up to 16) are read by the last MMA step
          const int n = (((valid + 15) & ~15) - valid) * 8;  // 16-byte words per box
          uint4* base = reinterpret_cast<uint4*>(stages + stage * W_STAGE) + valid * 8;
#pragma unroll
          for (int box = 0; box < 6; ++box)
            for (int i = lane; i < n; i += 32) base[box * (W_BOX / 16) + i] = make_uint4(0u, 0u, 0u, 0u);
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(ctl.masked(stage));
        }
        if (lane == 0) ptx::mbar_arrive(ctl.empty(stage));
        if (++stage == W_STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuer
      int stage = 0;
      uint32_t phase = 0, mpar = 0;  // mpar: per stage, parity of its next masked phase
      bool alive = true;
      int it = 0;
      for (int j = 0, tile; alive && (tile = sched_tile(j, blockIdx.x, gridDim.x, total, zig)) >= 0;
           ++j, ++it) {
        int e, m0, n0;
        decode_wtile(tile, MT, NT, n_fast, ord, e, m0, n0);
        const int rows = off[e + 1] - off[e];
        const int KB = (rows + WK - 1) / WK;
        const int buf = it & 1;
        const uint32_t aph = (it >> 1) & 1;
        if (!ctl.wait(ctl.acc_empty(buf), aph ^ 1u, 15)) {
          alive = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d = tmem_base + buf * WN;
        for (int kb = 0; kb < KB; ++kb) {
          const int valid = min(WK, rows - kb * WK);
          const bool tail = valid < WK;
          const bool ok = tail ? ctl.wait(ctl.masked(stage), mpar >> stage & 1u, 16)
                               : ctl.wait(ctl.full(stage), phase, 17);
          if (!ok) {
            alive = false;
            break;
          }
          if (tail) mpar ^= 1u << stage;
          ptx::tc_fence_after();
          const uint32_t a = ptx::smem_u32(stages + stage * W_STAGE);
          const uint32_t b = a + W_A_BYTES;
          const int steps = (valid + 15) >> 4;
#pragma unroll
          for (int s = 0; s < WK / 16; ++s) {
            if (s >= steps) break;
            // both MN-major: 64-wide chunks one box apart (LBO), 8-row K
            // groups 1 KB apart (SBO); a K step of 16 rows moves 2 KB
            const uint64_t adesc = ptx::sw128_desc(a + s * 2048, W_BOX, 1024);
            const uint64_t bdesc = ptx::sw128_desc(b + s * 2048, W_BOX, 1024);
            ptx::umma_bf16(d, adesc, bdesc, W_IDESC, (kb | s) != 0 ? 1u : 0u);
          }
          ptx::umma_commit(ctl.empty(stage));
          if (++stage == W_STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!alive) break;
        ptx::umma_commit(ctl.acc_full(buf));  // also for an expert without rows
      }
      if (!alive) {
        ptx::umma_commit(ctl.drain());
        ctl.wait(ctl.drain(), 0, 18, false);
      }
    }
  } else if (warp >= 2 && warp <= 5) {
    // ------------------------------------------------ epilogue warps 2..5
    const int q = warp & 3;
    const uint32_t stg = epi + q * 2 * W_STG_BYTES;
    uint32_t ck = 0;
    int it = 0;
    for (int j = 0, tile; (tile = sched_tile(j, blockIdx.x, gridDim.x, total, zig)) >= 0; ++j, ++it) {
      int e, m0, n0;
      decode_wtile(tile, MT, NT, n_fast, ord, e, m0, n0);
      const bool empty_expert = off[e + 1] == off[e];
      const int buf = it & 1;
      const uint32_t aph = (it >> 1) & 1;
      bool ok = ctl.wait(ctl.acc_full(buf), aph, 19);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      ptx::tc_fence_after();
      const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * WN;
      drain_to_tma(tb, &tmO, e * args.M + m0 + q * 32, n0, min(WN, args.N - n0), empty_expert, stg,
                   lane, ck);
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(ctl.acc_empty(buf));
    }
    if (lane == 0) ptx::bulk_wait_group_all();
  }
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, 512);
  }
}

// ------------------------------------------------------------------ SM pairs
// The same weight gradients on pairs of SMs (a 2-CTA cluster sharing each
// MMA, tcgen05 cta_group::2): tile = (expert, 256 rows of M, 256 columns of
// N), M=256,N=256,K=16 MMAs.  Rank r stages X's columns m0+128r..+127 (its
// accumulator rows) and Y's columns n0+128r..+127 (its half of B): a stage
// is two 64x64 boxes of each, 32 KB per CTA, 6 deep.  Each SM stages half of
// the B tile it multiplies by, as in the forward's pair kernel.
//  * Both CTAs' copies of a block count on one barrier in rank 0, armed by
//    rank 0 with both halves' bytes: `full` for a block inside the expert,
//    `tfull` for its last, partial block.  Each of the two completes once per
//    fill of its own kind, so its waiters keep a parity per stage (the ring
//    phase only describes `empty`, which every fill passes through).  Rank 0's seventh warp waits only
//    on `tfull` (phases complete in order, and the next tail fill of a stage
//    needs the MMA to have consumed this one, so no phase is skipped),
//    clears the rows up to the next 16-row MMA step in both CTAs' boxes (the
//    peer's through distributed shared memory), fences them for the tensor
//    core (fence.proxy.async.shared::cluster) and arrives on `masked`.
//  * Rank 0 issues the MMAs; its commits arrive on the empty/acc_full
//    barriers of both CTAs.  Each CTA's epilogue drains its 128 rows and
//    arrives on rank 0's acc_empty (8 arrivals).  When M % 256 == 128 the
//    last row tile's rank-1 half reads zeros (TMA fill) and stores nothing.
//  * A timed-out wait also raises the other CTA's abort flag; a CTA that
//    gives up waits (bounded) for the copies counted on its own barriers, or
//    pauses for the ones counted on its peer's; every cross-CTA access
//    happens before the final cluster barrier.
constexpr int PW_M = 256;                          // dW rows per pair tile
constexpr int PW_STAGE = 4 * W_BOX;                // 2 X boxes + 2 Y boxes: 32 KB
constexpr int PW_STAGES = 6;
constexpr int PW_NUM_BARS = 5 * PW_STAGES + 5;     // full, tfull, masked, empty, acc_*, drain
constexpr int PW_SMEM = 1024 + PW_STAGES * PW_STAGE + W_EPI_BYTES + PW_NUM_BARS * 8 + 16 +
                        (MOE_MAX_EXPERTS + 1) * 4 + MOE_MAX_EXPERTS;
static_assert(PW_SMEM <= 227 * 1024, "shared memory budget (pair)");
constexpr uint32_t PW_IDESC = ptx::idesc_bf16_f32(PW_M, WN, /*b_mn_major=*/true) | (1u << 15);
constexpr long long kPeerDrainCycles = 20000000LL;

struct PWCtl {
  uint64_t* bar;
  volatile int* abort_flag;
  int* err;
  uint32_t peer_abort;  // the other CTA's abort flag (shared::cluster)
  __device__ uint32_t full(int s) const { return ptx::smem_u32(bar + s); }
  __device__ uint32_t tfull(int s) const { return ptx::smem_u32(bar + PW_STAGES + s); }
  __device__ uint32_t masked(int s) const { return ptx::smem_u32(bar + 2 * PW_STAGES + s); }
  __device__ uint32_t empty(int s) const { return ptx::smem_u32(bar + 3 * PW_STAGES + s); }
  __device__ uint32_t acc_full(int b) const { return ptx::smem_u32(bar + 4 * PW_STAGES + b); }
  __device__ uint32_t acc_empty(int b) const { return ptx::smem_u32(bar + 4 * PW_STAGES + 2 + b); }
  __device__ uint32_t drain() const { return ptx::smem_u32(bar + 4 * PW_STAGES + 4); }
  __device__ bool wait(uint32_t b, uint32_t parity, int site, bool honour_abort = true) const {
    bool timed_out;
    if (ptx::mbar_wait_bounded(b, parity, kWaitCycles, abort_flag, honour_abort, &timed_out))
      return true;
    if (timed_out) {
      report_error(err, DEV_ERR_TIMEOUT, site);
      ptx::st_cluster_u32(peer_abort, 1u);
    }
    return false;
  }
};

__device__ __forceinline__ void st_cluster_zero16(uint32_t cluster_addr) {
  asm volatile("st.shared::cluster.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(cluster_addr), "r"(0u)
               : "memory");
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(W_THREADS, 1)
    tc_wgrad_pair_kernel(const __grid_constant__ CUtensorMap tmX,
                         const __grid_constant__ CUtensorMap tmY,
                         const __grid_constant__ CUtensorMap tmO, WgradArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* stages = smem;
  const uint32_t epi = ptx::smem_u32(smem + PW_STAGES * PW_STAGE);  // 1 KB aligned
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + PW_STAGES * PW_STAGE + W_EPI_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + PW_NUM_BARS);
  int* abort_word = reinterpret_cast<int*>(tmem_slot + 1);
  volatile int* abort_flag = abort_word;
  int* off = reinterpret_cast<int*>(tmem_slot + 4);
  uint8_t* ord = reinterpret_cast<uint8_t*>(off + MOE_MAX_EXPERTS + 1);
  int* zig_word = reinterpret_cast<int*>(tmem_slot + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  const int E = args.E;
  const int MT = (args.M + PW_M - 1) / PW_M, NT = (args.N + WN - 1) / WN;
  const int total = E * MT * NT;
  const bool n_fast = args.N < args.M;
  const PWCtl ctl{bars, abort_flag, args.err, ptx::mapa_shared(ptx::smem_u32(abort_word), rank ^ 1u)};

  if (threadIdx.x == 0) {
    for (int s = 0; s < PW_STAGES; ++s) {
      ptx::mbar_init(ctl.full(s), 1);
      ptx::mbar_init(ctl.tfull(s), 1);
      ptx::mbar_init(ctl.masked(s), 1);
      ptx::mbar_init(ctl.empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(ctl.acc_full(b), 1);
      ptx::mbar_init(ctl.acc_empty(b), 8);  // 4 epilogue warps in each CTA
    }
    ptx::mbar_init(ctl.drain(), 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
    ptx::prefetch_tensormap(&tmX);
    ptx::prefetch_tensormap(&tmY);
    ptx::prefetch_tensormap(&tmO);
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(ptx::smem_u32(tmem_slot), 512);
    ptx::tmem_relinquish_pair();
  }
  // no offsets: one dense group over rows [0, max_rows) (E == 1)
  for (int e = threadIdx.x; e <= E; e += blockDim.x)
    off[e] = args.offsets ? args.offsets[e] : (e == 0 ? 0 : static_cast<int>(args.max_rows));
  __syncthreads();
  if (threadIdx.x == 0) {  // offsets must start at 0, never decrease, end within the buffers
    bool ok = off[0] == 0 && off[E] <= args.max_rows;
    for (int e = 0; e < E; ++e) ok = ok && off[e + 1] >= off[e];
    if (!ok) {
      for (int e = 0; e <= E; ++e) off[e] = 0;
      if (blockIdx.x == 0) report_error(args.err, DEV_ERR_INDEX, -1);
    }
    int most = 0;
    for (int e = 0; e < E; ++e) most = max(most, off[e + 1] - off[e]);
    *zig_word = static_cast<int64_t>(most) * E > 4LL * off[E];
  }
  __syncthreads();
  const bool zig = *zig_word != 0;
  // skewed loads: experts by rows, most first (equal counts: lower index
  // first); balanced: index order
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int n = off[e + 1] - off[e];
    int r = e;
    if (zig) {
      r = 0;
      for (int q = 0; q < E; ++q) {
        const int m = off[q + 1] - off[q];
        r += (m > n) || (m == n && q < e);
      }
    }
    ord[r] = static_cast<uint8_t>(e);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();  // both CTAs' barriers initialised before any cross-CTA signal
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer (both CTAs)
      int stage = 0;
      uint32_t phase = 0;
      // per stage: filled, fill went to tfull, parity of the phase that
      // completes the latest fill, parity of the next full / tfull phase
      uint32_t filled = 0, tailbits = 0, fill_parity = 0, fnext = 0, tnext = 0;
      bool alive = true;
      for (int j = 0, tile; alive && (tile = sched_tile(j, pair, npairs, total, zig)) >= 0; ++j) {
        int e, m0, n0;
        decode_wtile(tile, MT, NT, n_fast, ord, e, m0, n0, PW_M);
        const int r0 = off[e], rows = off[e + 1] - off[e];
        const int KB = (rows + WK - 1) / WK;
        const int mx = m0 + static_cast<int>(rank) * 128, ny = n0 + static_cast<int>(rank) * 128;
        for (int kb = 0; kb < KB; ++kb) {
          if (!ctl.wait(ctl.empty(stage), phase ^ 1u, 21)) {
            alive = false;
            break;
          }
          const bool tail = rows - kb * WK < WK;
          const uint32_t bar = tail ? ctl.tfull(stage) : ctl.full(stage);
          if (rank == 0) ptx::mbar_arrive_expect_tx(bar, 2 * PW_STAGE);
          const uint32_t fb = ptx::mapa_shared(bar, 0);
          const uint32_t a = ptx::smem_u32(stages + stage * PW_STAGE);
          const uint32_t b = a + 2 * W_BOX;
          const int row = r0 + kb * WK;
          ptx::tma_load_2d_pair(a, &tmX, mx, row, fb);
          ptx::tma_load_2d_pair(a + W_BOX, &tmX, mx + 64, row, fb);
          ptx::tma_load_2d_pair(b, &tmY, ny, row, fb);
          ptx::tma_load_2d_pair(b + W_BOX, &tmY, ny + 64, row, fb);
          const uint32_t bit = 1u << stage;
          const uint32_t par = tail ? (tnext & bit) : (fnext & bit);
          if (tail)
            tnext ^= bit;
          else
            fnext ^= bit;
          filled |= bit;
          fill_parity = (fill_parity & ~bit) | par;
          tailbits = (tailbits & ~bit) | (tail ? bit : 0u);
          if (++stage == PW_STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (alive) {
        for (int i = 0; i < PW_STAGES; ++i) {
          if (!ctl.wait(ctl.empty(stage), phase ^ 1u, 22, false)) break;
          if (++stage == PW_STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      } else if (rank == 0) {
        // give up: wait (bounded) for the copies counted on this CTA's barriers
        for (int s = 0; s < PW_STAGES; ++s)
          if (filled >> s & 1u)
            ctl.wait((tailbits >> s & 1u) ? ctl.tfull(s) : ctl.full(s), fill_parity >> s & 1u, 23,
                     false);
      } else {
        // this CTA's copies complete on rank 0's barriers: pause (bounded)
        const long long t0 = clock64();
        while (clock64() - t0 < kPeerDrainCycles) {
        }
      }
    }
  } else if (warp == 6) {
    if (rank == 0) {
      // ------------------------------------------------ tail zeroing (rank 0, whole warp)
      int stage = 0;
      uint32_t tpar = 0;  // per stage: parity of its next tfull phase
      const uint32_t peer_stages = ptx::mapa_shared(ptx::smem_u32(stages), 1);
      for (int j = 0, tile; (tile = sched_tile(j, pair, npairs, total, zig)) >= 0; ++j) {
        int e, m0, n0;
        decode_wtile(tile, MT, NT, n_fast, ord, e, m0, n0, PW_M);
        const int rows = off[e + 1] - off[e];
        const int KB = (rows + WK - 1) / WK;
        bool alive = true;
        for (int kb = 0; kb < KB; ++kb) {
          const int valid = min(WK, rows - kb * WK);
          if (valid < WK) {
            if (!__all_sync(0xffffffffu, ctl.wait(ctl.tfull(stage), tpar >> stage & 1u, 24))) {
              alive = false;
              break;
            }
            tpar ^= 1u << stage;
            const int n = (((valid + 15) & ~15) - valid) * 8;  // 16-byte words per box
            const uint32_t off_bytes = stage * PW_STAGE + valid * 128;
            uint4* own = reinterpret_cast<uint4*>(stages + off_bytes);
#pragma unroll
            for (int box = 0; box < 4; ++box)
              for (int i = lane; i < n; i += 32) {
                own[box * (W_BOX / 16) + i] = make_uint4(0u, 0u, 0u, 0u);
                st_cluster_zero16(peer_stages + off_bytes + box * W_BOX + i * 16);
              }
            asm volatile("fence.proxy.async.shared::cluster;" ::: "memory");
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(ctl.masked(stage));
          }
          if (++stage == PW_STAGES) stage = 0;
        }
        if (!alive) break;
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ------------------------------------------------ MMA issuer (rank 0)
      int stage = 0;
      uint32_t fpar = 0, mpar = 0;  // per stage: parity of the next full / masked phase
      bool alive = true;
      int it = 0;
      for (int j = 0, tile; alive && (tile = sched_tile(j, pair, npairs, total, zig)) >= 0; ++j, ++it) {
        int e, m0, n0;
        decode_wtile(tile, MT, NT, n_fast, ord, e, m0, n0, PW_M);
        const int rows = off[e + 1] - off[e];
        const int KB = (rows + WK - 1) / WK;
        const int buf = it & 1;
        const uint32_t aph = (it >> 1) & 1;
        if (!ctl.wait(ctl.acc_empty(buf), aph ^ 1u, 25)) {
          alive = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d = tmem_base + buf * WN;
        for (int kb = 0; kb < KB; ++kb) {
          const int valid = min(WK, rows - kb * WK);
          const bool tail = valid < WK;
          const bool ok = tail ? ctl.wait(ctl.masked(stage), mpar >> stage & 1u, 26)
                               : ctl.wait(ctl.full(stage), fpar >> stage & 1u, 27);
          if (!ok) {
            alive = false;
            break;
          }
          if (tail)
            mpar ^= 1u << stage;
          else
            fpar ^= 1u << stage;
          ptx::tc_fence_after();
          const uint32_t a = ptx::smem_u32(stages + stage * PW_STAGE);
          const uint32_t b = a + 2 * W_BOX;
          const int steps = (valid + 15) >> 4;
#pragma unroll
          for (int s = 0; s < WK / 16; ++s) {
            if (s >= steps) break;
            // each CTA's halves: two 64-wide MN chunks one box apart (LBO),
            // 8-row K groups 1 KB apart (SBO), 2 KB per 16-row K step
            const uint64_t adesc = ptx::sw128_desc(a + s * 2048, W_BOX, 1024);
            const uint64_t bdesc = ptx::sw128_desc(b + s * 2048, W_BOX, 1024);
            ptx::umma_bf16_pair(d, adesc, bdesc, PW_IDESC, (kb | s) != 0 ? 1u : 0u);
          }
          ptx::umma_commit_pair(ctl.empty(stage), 3);
          if (++stage == PW_STAGES) stage = 0;
        }
        if (!alive) break;
        ptx::umma_commit_pair(ctl.acc_full(buf), 3);  // also for an expert without rows
      }
      if (!alive) {
        ptx::umma_commit_pair(ctl.drain(), 1);
        ctl.wait(ctl.drain(), 0, 28, false);
      }
    }
  } else if (warp >= 2 && warp <= 5) {
    // ------------------------------------------------ epilogue warps 2..5 (both CTAs)
    const int q = warp & 3;
    const uint32_t stg = epi + q * 2 * W_STG_BYTES;
    uint32_t ck = 0;
    int it = 0;
    for (int j = 0, tile; (tile = sched_tile(j, pair, npairs, total, zig)) >= 0; ++j, ++it) {
      int e, m0, n0;
      decode_wtile(tile, MT, NT, n_fast, ord, e, m0, n0, PW_M);
      const bool empty_expert = off[e + 1] == off[e];
      const int buf = it & 1;
      const uint32_t aph = (it >> 1) & 1;
      bool ok = ctl.wait(ctl.acc_full(buf), aph, 29);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      ptx::tc_fence_after();
      const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * WN;
      const int mbase = m0 + static_cast<int>(rank) * 128 + q * 32;  // lane l: row mbase + l
      if (mbase < args.M)
        drain_to_tma(tb, &tmO, e * args.M + mbase, n0, min(WN, args.N - n0), empty_expert, stg,
                     lane, ck);
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_cluster(ptx::mapa_shared(ctl.acc_empty(buf), 0));
    }
    if (lane == 0) ptx::bulk_wait_group_all();
  }
  __syncthreads();
  ptx::cluster_sync();  // no cross-CTA access after this point
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem_base, 512);
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

// [rows, cols] bf16 with row stride ld (elements), box 64 (cols) x 64 (rows)
bool map_mn(CUtensorMap* m, const void* ptr, int64_t cols, int64_t rows, int64_t ld) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
  cuuint32_t box[2] = {64, WK};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// dW [rows, N] fp32 (rows = E * M), box 32 (N) x 32 (rows), 128-byte swizzle:
// the epilogue's TMA stores.
bool map_out(CUtensorMap* m, float* ptr, int64_t N, int64_t rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(N) * 4};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, ptr, dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Pairs of SMs that can be resident at once for the pair kernel (0: none, or
// the query failed).
int wgrad_pair_slots() {
  static int cache[64] = {0};  // per device; -1 = queried, unusable
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (cache[dev] == 0) {
    int n = 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(W_THREADS, 1, 1);
    cfg.dynamicSmemBytes = PW_SMEM;
    if (cudaFuncSetAttribute(tc_wgrad_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             PW_SMEM) != cudaSuccess ||
        cudaOccupancyMaxActiveClusters(&n, tc_wgrad_pair_kernel, &cfg) != cudaSuccess || n <= 0) {
      cudaGetLastError();  // clear a failed query; the one-SM kernel is used instead
      n = -1;
    }
    cache[dev] = n;
  }
  return cache[dev] > 0 ? cache[dev] : 0;
}

}  // namespace

// SM pairs unless MOE_TC_PAIR=0 in the environment (a tuning override shared
// with the grouped GEMMs) or no 2-CTA cluster fits.
cudaError_t launch_tc_wgrad(int E, int M, int N, int64_t max_rows, const void* X, int ldx,
                            const void* Y, int ldy, const int32_t* offsets, float* dW, int* err,
                            cudaStream_t s) {
  if (E == 0) return cudaSuccess;
  if (M % WM != 0 || N % 128 != 0) return cudaErrorInvalidValue;
  if (offsets == nullptr && (E != 1 || max_rows > INT32_MAX)) return cudaErrorInvalidValue;
  const int64_t rows = max_rows > 0 ? max_rows : 1;  // a map needs a positive extent
  CUtensorMap mx, my, mo;
  if (!map_mn(&mx, X, M, rows, ldx) || !map_mn(&my, Y, N, rows, ldy) ||
      !map_out(&mo, dW, N, static_cast<int64_t>(E) * M))
    return cudaErrorInvalidValue;
  WgradArgs args{offsets, E, M, N, max_rows, dW, err};
  const char* force = getenv("MOE_TC_PAIR");
  const int slots = (force && force[0] == '0') ? 0 : wgrad_pair_slots();
  if (slots > 0) {
    const int64_t tiles = static_cast<int64_t>(E) * ((M + PW_M - 1) / PW_M) * ((N + WN - 1) / WN);
    const int64_t pairs = slots < tiles ? slots : tiles;
    tc_wgrad_pair_kernel<<<static_cast<unsigned>(2 * pairs), W_THREADS, PW_SMEM, s>>>(mx, my, mo,
                                                                                       args);
    return cudaGetLastError();
  }
  static bool configured[64] = {false};
  int dev = 0;
  cudaError_t st = cudaGetDevice(&dev);
  if (st != cudaSuccess) return st;
  if (dev < 64 && !configured[dev]) {
    st = cudaFuncSetAttribute(tc_wgrad_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, W_SMEM);
    if (st != cudaSuccess) return st;
    configured[dev] = true;
  }
  const int64_t tiles = static_cast<int64_t>(E) * (M / WM) * ((N + WN - 1) / WN);
  int64_t grid = device_sm_count();
  if (grid > tiles) grid = tiles;
  tc_wgrad_kernel<<<static_cast<unsigned>(grid), W_THREADS, W_SMEM, s>>>(mx, my, mo, args);
  return cudaGetLastError();
}

}  // namespace moe
