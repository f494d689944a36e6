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
//    expert; an expert with no rows gets a zero block.
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
//  * Every wait is bounded as in the forward kernel (error word, abort flag,
//    drain before TMEM is freed).
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
constexpr int W_PITCH = 36;
constexpr int W_EPI_BYTES = 4 * 32 * W_PITCH * 4;
constexpr int W_NUM_BARS = 3 * W_STAGES + 5;       // full, masked, empty, acc_full[2], acc_empty[2], drain
constexpr int W_SMEM = 1024 + W_STAGES * W_STAGE + W_EPI_BYTES + W_NUM_BARS * 8 + 16 +
                       (MOE_MAX_EXPERTS + 1) * 4;
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

__device__ __forceinline__ void decode_wtile(int tile, int MT, int NT, int& e, int& m0, int& n0) {
  e = tile / (MT * NT);
  const int u = tile - e * MT * NT;
  const int nt = u / MT;
  m0 = (u - nt * MT) * WM;
  n0 = nt * WN;
}

__global__ void __launch_bounds__(W_THREADS, 1)
    tc_wgrad_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmY,
                    WgradArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* stages = smem;
  float* epi = reinterpret_cast<float*>(smem + W_STAGES * W_STAGE);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + W_STAGES * W_STAGE + W_EPI_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + W_NUM_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* off = reinterpret_cast<int*>(tmem_slot + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = args.E;
  const int MT = args.M / WM, NT = (args.N + WN - 1) / WN;
  const int total = E * MT * NT;
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
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), 512);
    ptx::tmem_relinquish();
  }
  for (int e = threadIdx.x; e <= E; e += blockDim.x) off[e] = args.offsets[e];
  __syncthreads();
  if (threadIdx.x == 0) {  // offsets must start at 0, never decrease, end within the buffers
    bool ok = off[0] == 0 && off[E] <= args.max_rows;
    for (int e = 0; e < E; ++e) ok = ok && off[e + 1] >= off[e];
    if (!ok) {
      for (int e = 0; e <= E; ++e) off[e] = 0;
      if (blockIdx.x == 0) report_error(args.err, DEV_ERR_INDEX, -1);
    }
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
      for (int tile = blockIdx.x; alive && tile < total; tile += gridDim.x) {
        int e, m0, n0;
        decode_wtile(tile, MT, NT, e, m0, n0);
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
    for (int tile = blockIdx.x; alive && tile < total; tile += gridDim.x) {
      int e, m0, n0;
      decode_wtile(tile, MT, NT, e, m0, n0);
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
      for (int tile = blockIdx.x; alive && tile < total; tile += gridDim.x, ++it) {
        int e, m0, n0;
        decode_wtile(tile, MT, NT, e, m0, n0);
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
    float* etile = epi + q * (32 * W_PITCH);
    const int sub = lane >> 3, col4 = (lane & 7) * 4;
    int it = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++it) {
      int e, m0, n0;
      decode_wtile(tile, MT, NT, e, m0, n0);
      const bool empty_expert = off[e + 1] == off[e];
      const int buf = it & 1;
      const uint32_t aph = (it >> 1) & 1;
      bool ok = ctl.wait(ctl.acc_full(buf), aph, 19);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      ptx::tc_fence_after();
      const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * WN;
      const int mbase = m0 + q * 32;  // lane l holds output row mbase + l
      float* out0 = args.out + (static_cast<int64_t>(e) * args.M) * args.N + n0;
      const int valid = min(WN, args.N - n0);
#pragma unroll 1
      for (int c = 0; c < valid; c += 32) {
        uint32_t y[32];
        ptx::tmem_ld32(tb + c, y);
        ptx::tmem_wait_ld();
        float4* mine = reinterpret_cast<float4*>(etile + lane * W_PITCH);
#pragma unroll
        for (int v = 0; v < 8; ++v)
          mine[v] = empty_expert ? make_float4(0.f, 0.f, 0.f, 0.f)
                                 : make_float4(__uint_as_float(y[4 * v]), __uint_as_float(y[4 * v + 1]),
                                               __uint_as_float(y[4 * v + 2]), __uint_as_float(y[4 * v + 3]));
        __syncwarp();
#pragma unroll
        for (int r8 = 0; r8 < 8; ++r8) {
          const int r = r8 * 4 + sub;
          *reinterpret_cast<float4*>(out0 + static_cast<int64_t>(mbase + r) * args.N + c + col4) =
              *reinterpret_cast<const float4*>(etile + r * W_PITCH + col4);
        }
        __syncwarp();
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(ctl.acc_empty(buf));
    }
  }
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, 512);
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

}  // namespace

cudaError_t launch_tc_wgrad(int E, int M, int N, int64_t max_rows, const void* X, int ldx,
                            const void* Y, int ldy, const int32_t* offsets, float* dW, int* err,
                            cudaStream_t s) {
  if (E == 0) return cudaSuccess;
  if (M % WM != 0 || N % 128 != 0) return cudaErrorInvalidValue;
  const int64_t rows = max_rows > 0 ? max_rows : 1;  // a map needs a positive extent
  CUtensorMap mx, my;
  if (!map_mn(&mx, X, M, rows, ldx) || !map_mn(&my, Y, N, rows, ldy)) return cudaErrorInvalidValue;
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
  WgradArgs args{offsets, E, M, N, max_rows, dW, err};
  tc_wgrad_kernel<<<static_cast<unsigned>(grid), W_THREADS, W_SMEM, s>>>(mx, my, args);
  return cudaGetLastError();
}

}  // namespace moe
