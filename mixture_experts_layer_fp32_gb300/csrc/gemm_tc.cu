// bf16 grouped expert MLP on the 5th-generation tensor cores (tcgen05).
//
// Grouped expert MLP of §10 of "MoE我们喜欢你（三）：Megatron Core MoE 源码路径解析"
// (r00kie-liu.github.io): all local experts' GEMMs in one launch
// (TEGroupedMLP / GroupedLinear on that page), with SwiGLU experts:
//   fc1:  H[r, :] = silu(X[r, :] . W1[e]) * (X[r, :] . W3[e])   (bf16 out)
//   fc2:  Y[r, :] = H[r, :] . W2[e]                              (fp32 out)
// for the rows r of expert e, [offsets[e], offsets[e+1]).  With no offsets
// array the launch is one dense group (E = 1) over rows [0, max_rows): the
// shared expert, applied to every token.
//
// Design (one CTA per SM, persistent):
//  * Output tile 128 rows x 256 fp32 accumulator columns in TMEM.  fc1's
//    256 columns are 128 columns of W1 next to the same 128 columns of W3,
//    so one M=128,N=256,K=16 MMA produces both halves of the SwiGLU and the
//    epilogue pairs column j with column 128+j.  fc2's 256 columns are 256
//    columns of W2.
//  * The tile list is built on the device from the expert offsets (written
//    by the permutation kernel): expert e owns ceil(rows_e/128) row blocks x
//    n-tiles, the smaller side inner (row blocks, unless the expert has
//    more rows than accumulator columns) so that CTAs running together share
//    the re-read operand through L2.  No host synchronisation.
//  * Warp roles: warp 0 lane 0 issues TMA loads (A tile 128x64 and four
//    64xBK weight boxes per stage; a 4-deep ring of K=64 stages), warp 1
//    allocates TMEM and lane 0 issues tcgen05.mma, warps 2-5 drain TMEM with
//    tcgen05.ld, apply the epilogue and store (warps 2-9 in the E4M3 fc1,
//    two per TMEM lane quarter, each half the columns).  Two accumulator buffers
//    (2 x 256 of the 512 TMEM columns) overlap the epilogue of one tile with
//    the main loop of the next.
//  * A tile's rows past its expert's end are computed but never stored;
//    rows past the buffer end are zero-filled by TMA.
//  * Weights stay in the caller's [E, K, N] layout (N contiguous): the B
//    operand is MN-major in shared memory.  Activations are K-major.
//  * E4M3 variant (template flag FP8; the FP8 experts): both operands are
//    E4M3 codes and K-major (the weights are quantised once into [E, N, K]),
//    a stage carries 128 K values (the same 128-byte swizzled rows), the MMA
//    is kind::f8f6f4 with K = 32, and the epilogue multiplies the fp32
//    accumulator by the row scale and the output channel's scale.
//  * tc_grouped_pair_kernel (below) runs the same tiles on pairs of SMs.
//  * Every wait is bounded: after ~2 s without progress the CTA records
//    MOE_ERR_TIMEOUT in the workspace error word, lets its in-flight copies
//    and MMAs finish (again bounded), frees its TMEM and exits.
#include <stdlib.h>

#include "common.cuh"
#include "sm100_ptx.cuh"

namespace moe {
namespace {

constexpr int BM = 128;
constexpr int BN = 256;                      // MMA N = accumulator columns
// K per pipeline stage.  64 (the default) gives 48 KB stages and a 4-deep
// ring; 32 (bf16 forward modes only) gives 24 KB stages and an 8-deep ring.
// Measured on GB300: 32 is 30-45% slower on every workload (Mixtral fc1 2170
// -> 3088 us, Switch fc1 445 -> 572 us): twice the per-stage barrier and TMA
// work and half-width A rows outweigh the deeper ring.
#ifndef MOE_TC_BK
#define MOE_TC_BK 64
#endif
constexpr int BK = MOE_TC_BK;
static_assert(BK == 32 || BK == 64, "K per stage");
constexpr int A_BYTES = BM * BK * 2;         // BK=32: 8 KB (64-byte rows, 64-byte swizzle)
constexpr int BOX_BYTES = 64 * BK * 2;       // 64 (N) x BK (K) weight box, 128-byte swizzle
constexpr int B_BYTES = 4 * BOX_BYTES;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int SMEM_BUDGET = 227 * 1024;
constexpr uint32_t A_LAYOUT = (BK == 64) ? ptx::kLayoutSw128 : ptx::kLayoutSw64;
constexpr uint32_t A_SBO = 8 * BK * 2;       // 8-row groups of A
constexpr int ACC_COLS = BN;
constexpr uint32_t TMEM_COLS = 512;
constexpr int THREADS = 192;
// fp32-output epilogue staging, per epilogue warp a 5 KB region (1 KB
// aligned): a 32 x 32 fp32 block in the 128-byte swizzle that a TMA store
// reads, or, for a warp whose rows cross the expert's end, a 32 x 32 tile
// with rows padded to 36 floats for masked row-segment stores (16-byte
// accesses of a quarter-warp hit distinct banks).
constexpr int EPI_PITCH = 36;
constexpr int EPI_WARP_BYTES = 5120;
constexpr int EPI_BYTES = 4 * EPI_WARP_BYTES;
static_assert(32 * EPI_PITCH * 4 <= EPI_WARP_BYTES && 4096 <= EPI_WARP_BYTES, "staging");
// the ring takes what the alignment slack, the epilogue staging and ~4 KB of
// barriers and offsets leave: 8 stages (BK=32) or 4 (BK=64)
constexpr int STAGES = (SMEM_BUDGET - 1024 - EPI_BYTES - 4096) / STAGE_BYTES;
constexpr int NUM_BARS = 2 * STAGES + 5;     // full, empty, acc_full[2], acc_empty[2], drain
constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + EPI_BYTES + NUM_BARS * 8 + 16 +
                           2 * (MOE_MAX_EXPERTS + 1) * 4;
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
constexpr uint32_t IDESC = ptx::idesc_bf16_f32(BM, BN, /*b_mn_major=*/true);
// E4M3 operands: a stage holds 128 K values (128 bytes per row, the same
// bytes as 64 bf16), the MMA takes K = 32, and B is K-major (one row of
// 128 bytes per output channel), 128-row boxes of 16 KB.
constexpr int KE_FP8 = 128;
constexpr uint32_t IDESC_F8 = ptx::idesc_e4m3_f32(BM, BN);
// bf16 with B K-major (the backward's dgrad GEMMs)
constexpr uint32_t IDESC_KB = ptx::idesc_bf16_f32(BM, BN, /*b_mn_major=*/false);
constexpr long long kWaitCycles = 4000000000LL;

// Forward modes FC1 (SwiGLU, bf16 out) and FC2 (fp32 out); backward modes:
//   FC1_BWD    the FC1 mainloop recomputes a = X.W1 and g = X.W3; the epilogue
//              reads dH and writes da = dH g silu'(a) and dg = dH silu(a)
//              (bf16) side by side into rows of 2f: [da | dg]
//   DGRAD_BF16 C = A . B^T with B K-major (a weight read in place, one row per
//              output column), bf16 out: fc2's dH = dY . W2[e]^T
//   DGRAD_F32  the same with K split between two weights (the first kb_split
//              K blocks from tmB0, the rest from tmB1), fp32 out: fc1's
//              dX = [da | dg] . [W1[e] ; W3[e]]^T
//   FC2_Y      fc2 of a top-1 layer with the combine in its epilogue: row r
//              is the one slot of token row_token[r], whose output row gets
//              bf16(row_weight[r] * acc) -- the combine's arithmetic, so the
//              bits equal fc2 followed by the combine kernel
//   FC2_F16S   fc2 with y_perm stored as fp16 plus one power-of-two scale per 32
//              columns (a row's chunk scaled so that its largest magnitude lands
//              in [2^14, 2^15)): 2 bytes per value instead of 4, relative error
//              2^-11 instead of 2^-24
enum { FC1 = 0, FC2 = 1, FC1_BWD = 2, DGRAD_BF16 = 3, DGRAD_F32 = 4, FC2_Y = 5, FC2_F16S = 6 };

// The one-SM kernel's E4M3 fc1 drains each accumulator with two warps per
// TMEM lane quarter (each takes half the output columns): with K = 1024 the
// scaled SwiGLU epilogue of four warps took longer than a tile's mainloop,
// which runs twice as fast as in bf16.
template <int MODE, bool FP8>
__host__ __device__ constexpr int epi_warps() {
  return MODE == FC1 && FP8 ? 8 : 4;
}
template <int MODE, bool FP8>
__host__ __device__ constexpr int one_sm_threads() {
  return 64 + 32 * epi_warps<MODE, FP8>();
}

// Exponent of the power-of-two scale of a 32-value chunk whose largest
// magnitude is amax: amax * 2^-e lies in [2^14, 2^15) for normal amax (e from
// the float's exponent field, clamped so that 2^-e and 2^e are normal floats);
// 0 for a non-finite amax (the values pass through the conversion unchanged).
__device__ __forceinline__ int f16s_exponent(float amax) {
  const int be = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFFu);
  if (be == 0xFF) return 0;
  const int e = be - 127 - 14;
  return e < -126 ? -126 : e;
}

struct TcArgs {
  const int32_t* offsets;
  int E;
  int num_n_tiles;
  int k_blocks;
  int64_t max_rows;
  void* out;
  int ldo;
  int* err;
  // E4M3 operands only: A row r's scale is row_scale[row_src ? row_src[r] : r];
  // output channel n of expert e has scale col_scale0[e * ncols + n] (W1 or W2)
  // and, for fc1's gate half, col_scale1[e * ncols + n] (W3)
  const float* row_scale = nullptr;
  const int32_t* row_src = nullptr;
  const float* col_scale0 = nullptr;
  const float* col_scale1 = nullptr;
  int ncols = 0;
  // FC1_BWD: dH [rows, ncols] bf16 (row stride ldaux); DGRAD_F32: K blocks
  // taken from tmB0 before tmB1
  const void* aux = nullptr;
  int ldaux = 0;
  int kb_split = 0;
  // DGRAD_F32: add to the output instead of overwriting it
  int accumulate = 0;
  // FC2 / DGRAD_F32 without accumulate: fp32 output rows stored by TMA
  // through the output tensor map (32 x 32 boxes) when a warp's 32 rows all
  // belong to the tile's expert
  int tma_out = 0;
  // FC2_Y: the token of each row (-1: none) and its combine weight
  const int32_t* row_token = nullptr;
  const float* row_weight = nullptr;
  // FC2_F16S: the chunk exponents [rows, ldo / 32] int8 (the fp16 values go to out)
  int8_t* exp_out = nullptr;
  // DGRAD_F32 with piece_cols > 0 (the router's logits over the split gate
  // weights): output column n goes to column n % piece_cols of partial
  // n / piece_cols, partials [num_pieces][rows][piece_cols] piece_stride
  // floats apart; columns of pieces >= num_pieces are not stored
  int piece_cols = 0;
  int num_pieces = 0;
  int64_t piece_stride = 0;
  // DGRAD_F32, dense A split along K (ksplit != 0, offsets == nullptr): group
  // e is K blocks [e * k_blocks, (e + 1) * k_blocks) of the same A rows, its
  // output rows the virtual rows [e * R, (e + 1) * R) with R = max_rows / E;
  // the weight is the map's first (and only) matrix
  int ksplit = 0;
};

// Barriers of an NS-stage ring: full[NS], empty[NS], acc_full[2],
// acc_empty[2], drain.
template <int NS>
struct CtlN {
  uint64_t* bar;
  volatile int* abort_flag;
  int* err;
  uint32_t peer_abort = 0;  // pair kernel: the other CTA's abort flag (shared::cluster)
  __device__ uint32_t full(int s) const { return ptx::smem_u32(bar + s); }
  __device__ uint32_t empty(int s) const { return ptx::smem_u32(bar + NS + s); }
  __device__ uint32_t acc_full(int b) const { return ptx::smem_u32(bar + 2 * NS + b); }
  __device__ uint32_t acc_empty(int b) const { return ptx::smem_u32(bar + 2 * NS + 2 + b); }
  __device__ uint32_t drain() const { return ptx::smem_u32(bar + 2 * NS + 4); }

  // Bounded wait.  Returns false on timeout (recorded) or, when
  // `honour_abort`, as soon as another role has given up.
  __device__ bool wait(uint32_t b, uint32_t parity, int site, bool honour_abort = true) const {
    bool timed_out;
    if (ptx::mbar_wait_bounded(b, parity, kWaitCycles, abort_flag, honour_abort, &timed_out))
      return true;
    if (timed_out) {
      report_error(err, DEV_ERR_TIMEOUT, site);
      if (peer_abort) ptx::st_cluster_u32(peer_abort, 1u);
    }
    return false;
  }
};
using Ctl = CtlN<STAGES>;

// Tile `tile` of the device-built list: expert e, first row m0 of its row
// block (ROWS rows per block), the expert's row end, and the n-tile.
// Inside an expert the smaller side varies fastest, so that the ~150 tiles in
// flight share the operand that is re-read: with fewer rows than accumulator
// columns (NT x BN) the row blocks are inner and the CTAs in flight share one
// weight n-tile while the expert's rows stay in L2; with more rows (an expert
// holding a large share of the tokens) the n-tiles are inner, the expert's
// weights stay in L2 and its rows stream once (row blocks inner would read
// them once per n-tile).
template <int ROWS = BM>
__device__ __forceinline__ void decode_tile(int tile, const int* tstart, const int* off, int E,
                                            int NT, int& e, int& m0, int& rend, int& nt) {
  int lo = 0, hi = E;  // largest e in [0, E) with tstart[e] <= tile
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (tstart[mid] <= tile) lo = mid; else hi = mid;
  }
  e = lo;
  const int rows = off[e + 1] - off[e];
  const int mt = (rows + ROWS - 1) / ROWS;
  const int u = tile - tstart[e];
  int rb;
  if (rows > NT * BN) {
    rb = u / NT;
    nt = u - rb * NT;
  } else {
    nt = u / mt;
    rb = u - nt * mt;
  }
  m0 = off[e] + rb * ROWS;
  rend = off[e + 1];
}

// Expert offsets into shared memory.  Without an offsets array (dense
// mode) the E groups are max_rows / E rows each (E = 1: rows [0, max_rows);
// E > 1: the K splits of a dense GEMM).
__device__ __forceinline__ void load_offsets(int* off, const TcArgs& args) {
  for (int e = threadIdx.x; e <= args.E; e += blockDim.x)
    off[e] = args.offsets ? args.offsets[e]
                          : static_cast<int>(static_cast<int64_t>(e) * (args.max_rows / args.E));
}

// Per-expert tile prefix (tstart[0..E]) from the expert offsets, by warp 0:
// expert e owns ceil(rows_e / ROWS) x NT tiles.  Inconsistent offsets (not
// starting at 0, decreasing, or past max_rows) give an empty list and a
// recorded device error.
template <int ROWS>
__device__ __forceinline__ void build_tile_prefix(const int* off, int* tstart, int E, int NT,
                                                  int64_t max_rows, int* err, int lane) {
  constexpr int PER = MOE_MAX_EXPERTS / 32;  // lane handles experts [8*lane, 8*lane + 8)
  int v[PER];
  int run = 0;
  bool ok = true;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int e = lane * PER + i;
    int t = 0;
    if (e < E) {
      const int rows = off[e + 1] - off[e];
      ok = ok && rows >= 0;
      t = ((rows + ROWS - 1) / ROWS) * NT;
    }
    v[i] = t;
    run += t;
  }
  if (lane == 0) ok = ok && off[0] == 0 && static_cast<int64_t>(off[E]) <= max_rows;
  ok = __all_sync(0xffffffffu, ok);
  int incl = run;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  int excl = incl - run;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int e = lane * PER + i;
    if (e < E) tstart[e] = ok ? excl : 0;
    excl += v[i];
  }
  if (lane == 31) tstart[E] = ok ? excl : 0;
  if (!ok && lane == 0 && blockIdx.x == 0) report_error(err, DEV_ERR_INDEX, -1);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// silu(a) * g with the approximate divide (a times the hardware reciprocal
// of 1 + e^-a, within 2 ulp of fp32; 0 once e^-a overflows): the rounding
// to bf16 that follows is 2^-9 relative.  The IEEE division's longer
// instruction sequence made the fc1 epilogue outlast a K = 1024 mainloop.
__device__ __forceinline__ float silu_mul(float a, float g) {
  return __fdividef(a, 1.0f + __expf(-a)) * g;
}

// Drain one accumulator buffer into the output: this warp's 32 TMEM lanes at
// `tb` hold rows rbase .. rbase+31 (lane l holds row rbase + l) of a tile of
// n-tile `nt`; rows at or past `rend` belong to no row of this expert and are
// not stored.  fc1 applies silu(a) * g and stores bf16, fc2 stores fp32.
// ch >= 0 (E4M3 fc1 on one SM, two warps per lane quarter): the warp drains
// output columns 64*ch .. 64*ch+63 of the n-tile only.
__device__ __forceinline__ void st_shared_v4(uint32_t a, uint32_t x, uint32_t y, uint32_t z,
                                             uint32_t w) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(x), "r"(y), "r"(z), "r"(w)
               : "memory");
}

template <int MODE, bool FP8>
__device__ __forceinline__ void drain_accumulator(uint32_t tb, float* etile, uint32_t stg,
                                                  const CUtensorMap* tmC, int rbase, int rend,
                                                  int nt, int e, const TcArgs& args, int lane,
                                                  int ch = -1) {
  const int sub = lane >> 3;
  const int col4 = (lane & 7) * 4;
  // E4M3: this lane's row scale (rows past the expert's end are not read)
  float rs = 1.f;
  if (FP8 && rbase + lane < rend) {
    const int r = rbase + lane;
    rs = args.row_scale[args.row_src ? args.row_src[r] : r];
  }
  if (MODE == FC1) {
    // silu(a) * g, packed to bf16: each lane writes 64 contiguous bytes
    // of its own row per 32-column chunk (whole 32-byte sectors; staging
    // through shared memory as fc2 does was measured slower here).
    const int row = rbase + lane;
    const int npair = ch >= 0 ? BN / 4 : BN / 2;  // output columns of this warp
    const int cofs = ch >= 0 ? ch * (BN / 4) : 0;  // and the first of them
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(args.out) +
                         static_cast<int64_t>(row) * args.ldo + nt * (BN / 2) + cofs;
#pragma unroll 1
    for (int c = 0; c < npair; c += 32) {
      uint32_t a[32], g[32];
      ptx::tmem_ld32(tb + cofs + c, a);
      ptx::tmem_ld32(tb + BN / 2 + cofs + c, g);
      ptx::tmem_wait_ld();
      if (row < rend) {
        uint4* dst = reinterpret_cast<uint4*>(out + c);
        if (FP8) {  // acc * row scale * channel scale (W1 half and W3 half)
          const int64_t cb = static_cast<int64_t>(e) * args.ncols + nt * (BN / 2) + cofs + c;
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            const float4 u = __ldg(reinterpret_cast<const float4*>(args.col_scale0 + cb + j));
            const float4 v = __ldg(reinterpret_cast<const float4*>(args.col_scale1 + cb + j));
            a[j] = __float_as_uint(__uint_as_float(a[j]) * (rs * u.x));
            a[j + 1] = __float_as_uint(__uint_as_float(a[j + 1]) * (rs * u.y));
            a[j + 2] = __float_as_uint(__uint_as_float(a[j + 2]) * (rs * u.z));
            a[j + 3] = __float_as_uint(__uint_as_float(a[j + 3]) * (rs * u.w));
            g[j] = __float_as_uint(__uint_as_float(g[j]) * (rs * v.x));
            g[j + 1] = __float_as_uint(__uint_as_float(g[j + 1]) * (rs * v.y));
            g[j + 2] = __float_as_uint(__uint_as_float(g[j + 2]) * (rs * v.z));
            g[j + 3] = __float_as_uint(__uint_as_float(g[j + 3]) * (rs * v.w));
          }
        }
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          uint4 w;
          w.x = pack_bf16x2(silu_mul(__uint_as_float(a[8 * v + 0]), __uint_as_float(g[8 * v + 0])),
                            silu_mul(__uint_as_float(a[8 * v + 1]), __uint_as_float(g[8 * v + 1])));
          w.y = pack_bf16x2(silu_mul(__uint_as_float(a[8 * v + 2]), __uint_as_float(g[8 * v + 2])),
                            silu_mul(__uint_as_float(a[8 * v + 3]), __uint_as_float(g[8 * v + 3])));
          w.z = pack_bf16x2(silu_mul(__uint_as_float(a[8 * v + 4]), __uint_as_float(g[8 * v + 4])),
                            silu_mul(__uint_as_float(a[8 * v + 5]), __uint_as_float(g[8 * v + 5])));
          w.w = pack_bf16x2(silu_mul(__uint_as_float(a[8 * v + 6]), __uint_as_float(g[8 * v + 6])),
                            silu_mul(__uint_as_float(a[8 * v + 7]), __uint_as_float(g[8 * v + 7])));
          dst[v] = w;
        }
      }
    }
  } else if (MODE == FC1_BWD) {
    // SwiGLU backward on the recomputed a (columns 0..127) and g (128..255):
    // each lane reads its row's 32 dH values per chunk (64 contiguous
    // bytes) and writes 64 bytes of da and of dg.
    const int row = rbase + lane;
    const int64_t col0 = static_cast<int64_t>(nt) * (BN / 2);
    const __nv_bfloat16* dh = static_cast<const __nv_bfloat16*>(args.aux) +
                              static_cast<int64_t>(row) * args.ldaux + col0;
    __nv_bfloat16* da_out = static_cast<__nv_bfloat16*>(args.out) +
                            static_cast<int64_t>(row) * args.ldo + col0;
    __nv_bfloat16* dg_out = da_out + args.ncols;
#pragma unroll 1
    for (int c = 0; c < BN / 2; c += 32) {
      uint32_t a[32], g[32];
      ptx::tmem_ld32(tb + c, a);
      ptx::tmem_ld32(tb + BN / 2 + c, g);
      ptx::tmem_wait_ld();
      if (row < rend) {
        const uint4* src = reinterpret_cast<const uint4*>(dh + c);
        uint4* dst_a = reinterpret_cast<uint4*>(da_out + c);
        uint4* dst_g = reinterpret_cast<uint4*>(dg_out + c);
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const uint4 hv = src[v];
          const uint32_t hw[4] = {hv.x, hv.y, hv.z, hv.w};
          uint32_t oa[4], og[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            float r_a[2], r_g[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const int j = 8 * v + 2 * q + u;
              const float dH = __uint_as_float(u ? (hw[q] & 0xffff0000u) : (hw[q] << 16));
              const float av = __uint_as_float(a[j]), gv = __uint_as_float(g[j]);
              const float sg = __fdividef(1.0f, 1.0f + __expf(-av));  // as silu_mul
              r_a[u] = dH * gv * (sg * (1.0f + av * (1.0f - sg)));
              r_g[u] = dH * (av * sg);
            }
            oa[q] = pack_bf16x2(r_a[0], r_a[1]);
            og[q] = pack_bf16x2(r_g[0], r_g[1]);
          }
          dst_a[v] = make_uint4(oa[0], oa[1], oa[2], oa[3]);
          dst_g[v] = make_uint4(og[0], og[1], og[2], og[3]);
        }
      }
    }
  } else if (MODE == FC2_Y) {
    // the top-1 combine: this lane's row goes, weighted, to its token's output
    // row (64 contiguous bytes per 32-column chunk); fmaf(w, acc, 0) is the
    // combine kernel's first (and, for one slot, only) step
    const int row = rbase + lane;
    int tok = -1;
    float w = 0.f;
    if (row < rend) {
      tok = args.row_token[row];
      w = args.row_weight[row];
    }
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(args.out) +
                         static_cast<int64_t>(tok < 0 ? 0 : tok) * args.ldo +
                         static_cast<int64_t>(nt) * BN;
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
      uint32_t y[32];
      ptx::tmem_ld32(tb + c, y);
      ptx::tmem_wait_ld();
      if (tok >= 0) {
        float v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(y[j]);
        if (FP8) {  // acc * row scale * channel scale, as fc2 stores it
          const float* cs = args.col_scale0 + static_cast<int64_t>(e) * args.ncols + nt * BN + c;
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const float4 u = __ldg(reinterpret_cast<const float4*>(cs + 4 * q));
            v[4 * q] *= rs * u.x;
            v[4 * q + 1] *= rs * u.y;
            v[4 * q + 2] *= rs * u.z;
            v[4 * q + 3] *= rs * u.w;
          }
        }
        uint4* dst = reinterpret_cast<uint4*>(out + c);
#pragma unroll
        for (int q = 0; q < 4; ++q)
          dst[q] = make_uint4(pack_bf16x2(fmaf(w, v[8 * q], 0.f), fmaf(w, v[8 * q + 1], 0.f)),
                              pack_bf16x2(fmaf(w, v[8 * q + 2], 0.f), fmaf(w, v[8 * q + 3], 0.f)),
                              pack_bf16x2(fmaf(w, v[8 * q + 4], 0.f), fmaf(w, v[8 * q + 5], 0.f)),
                              pack_bf16x2(fmaf(w, v[8 * q + 6], 0.f), fmaf(w, v[8 * q + 7], 0.f)));
      }
    }
  } else if (MODE == FC2_F16S) {
    // each lane's row, 32 columns at a time: the chunk's exponent from its
    // largest magnitude, the values times 2^-e (exact) rounded to fp16, and
    // one exponent byte per chunk (the row's 8 of this n-tile stored together)
    const int row = rbase + lane;
    int8_t* ex = args.exp_out + static_cast<int64_t>(row) * (args.ldo / 32) + nt * (BN / 32);
    uint32_t ex_lo = 0, ex_hi = 0;
    if (args.tma_out) {
      if (lane == 0) ptx::bulk_wait_group_read<0>();  // the staging block is free
      __syncwarp();
    }
    if (args.tma_out && rbase + 32 <= rend) {
      // every row of the warp is the expert's: 64 columns (two chunks) at a
      // time, 32 rows x 128 bytes of fp16 in the 128-byte swizzle (16-byte
      // piece j of row l at piece j ^ (l & 7)), one TMA store from lane 0
#pragma unroll 1
      for (int c = 0; c < BN; c += 64) {
        uint32_t y[2][32];
        ptx::tmem_ld32(tb + c, y[0]);
        ptx::tmem_ld32(tb + c + 32, y[1]);
        ptx::tmem_wait_ld();
        uint32_t hw[32];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          float v[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(y[half][j]);
          if (FP8) {  // acc * row scale * channel scale, as fc2 stores it
            const float* cs =
                args.col_scale0 + static_cast<int64_t>(e) * args.ncols + nt * BN + c + 32 * half;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const float4 u = __ldg(reinterpret_cast<const float4*>(cs + 4 * q));
              v[4 * q] *= rs * u.x;
              v[4 * q + 1] *= rs * u.y;
              v[4 * q + 2] *= rs * u.z;
              v[4 * q + 3] *= rs * u.w;
            }
          }
          float amax = 0.f;
#pragma unroll
          for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(v[j]));
          const int e8 = f16s_exponent(amax);
          const float down = __uint_as_float(static_cast<uint32_t>(127 - e8) << 23);  // 2^-e
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            __half2 hv = __floats2half2_rn(v[2 * j] * down, v[2 * j + 1] * down);
            hw[16 * half + j] = *reinterpret_cast<uint32_t*>(&hv);
          }
          const int cc = c + 32 * half;  // chunk cc/32 at byte cc/32 of the 8
          const uint32_t byte = static_cast<uint32_t>(e8) & 0xFFu;
          if (cc < 128) ex_lo |= byte << (cc / 4);
          else ex_hi |= byte << ((cc - 128) / 4);
        }
        if (c > 0) {
          if (lane == 0) ptx::bulk_wait_group_read<0>();
          __syncwarp();
        }
        const uint32_t srow = stg + lane * 128;
#pragma unroll
        for (int j = 0; j < 8; ++j)
          st_shared_v4(srow + ((j ^ (lane & 7)) << 4), hw[4 * j], hw[4 * j + 1], hw[4 * j + 2],
                       hw[4 * j + 3]);
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          ptx::tma_store_2d(tmC, nt * BN + c, rbase, stg);
          ptx::bulk_commit_group();
        }
      }
      *reinterpret_cast<uint2*>(ex) = make_uint2(ex_lo, ex_hi);
      return;
    }
    __half* out = static_cast<__half*>(args.out) + static_cast<int64_t>(row) * args.ldo +
                  static_cast<int64_t>(nt) * BN;
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
      uint32_t y[32];
      ptx::tmem_ld32(tb + c, y);
      ptx::tmem_wait_ld();
      if (row < rend) {
        float v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(y[j]);
        if (FP8) {  // acc * row scale * channel scale, as fc2 stores it
          const float* cs = args.col_scale0 + static_cast<int64_t>(e) * args.ncols + nt * BN + c;
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const float4 u = __ldg(reinterpret_cast<const float4*>(cs + 4 * q));
            v[4 * q] *= rs * u.x;
            v[4 * q + 1] *= rs * u.y;
            v[4 * q + 2] *= rs * u.z;
            v[4 * q + 3] *= rs * u.w;
          }
        }
        float amax = 0.f;
#pragma unroll
        for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(v[j]));
        const int e8 = f16s_exponent(amax);
        const float down = __uint_as_float(static_cast<uint32_t>(127 - e8) << 23);  // 2^-e
        uint32_t hw[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          __half2 hv = __floats2half2_rn(v[2 * j] * down, v[2 * j + 1] * down);
          hw[j] = *reinterpret_cast<uint32_t*>(&hv);
        }
        uint4* dst = reinterpret_cast<uint4*>(out + c);
#pragma unroll
        for (int q = 0; q < 4; ++q)
          dst[q] = make_uint4(hw[4 * q], hw[4 * q + 1], hw[4 * q + 2], hw[4 * q + 3]);
        const uint32_t byte = static_cast<uint32_t>(e8) & 0xFFu;
        if (c < 128) ex_lo |= byte << (c / 4);  // chunk c/32 at bit 8 * (c/32)
        else ex_hi |= byte << ((c - 128) / 4);
      }
    }
    if (row < rend) *reinterpret_cast<uint2*>(ex) = make_uint2(ex_lo, ex_hi);
  } else if (MODE == DGRAD_BF16) {
    // plain bf16 output, 256 columns: each lane writes 64 bytes of its row per
    // chunk; chunks at or past ncols (the last tile when ncols % 256 == 128)
    // are not stored
    const int row = rbase + lane;
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(args.out) +
                         static_cast<int64_t>(row) * args.ldo + static_cast<int64_t>(nt) * BN;
    const int valid = min(BN, args.ncols - nt * BN);
#pragma unroll 1
    for (int c = 0; c < valid; c += 32) {
      uint32_t y[32];
      ptx::tmem_ld32(tb + c, y);
      ptx::tmem_wait_ld();
      if (row < rend) {
        uint4* dst = reinterpret_cast<uint4*>(out + c);
#pragma unroll
        for (int v = 0; v < 4; ++v)
          dst[v] = make_uint4(
              pack_bf16x2(__uint_as_float(y[8 * v]), __uint_as_float(y[8 * v + 1])),
              pack_bf16x2(__uint_as_float(y[8 * v + 2]), __uint_as_float(y[8 * v + 3])),
              pack_bf16x2(__uint_as_float(y[8 * v + 4]), __uint_as_float(y[8 * v + 5])),
              pack_bf16x2(__uint_as_float(y[8 * v + 6]), __uint_as_float(y[8 * v + 7])));
      }
    }
  } else {
    // the warp's staging region is free once its last TMA store has read it
    if (args.tma_out) {
      if (lane == 0) ptx::bulk_wait_group_read<0>();
      __syncwarp();
    }
    if (args.tma_out && !(MODE == DGRAD_F32 && args.accumulate) && rbase + 32 <= rend) {
      // every row of the warp is the expert's: 32 x 32 blocks in the
      // 128-byte swizzle (16-byte chunk j of row l at chunk j ^ (l & 7)),
      // one TMA store each from lane 0
#pragma unroll 1
      for (int c = 0; c < BN; c += 32) {
        uint32_t y[32];
        ptx::tmem_ld32(tb + c, y);
        ptx::tmem_wait_ld();
        if (FP8) {  // acc * row scale * channel scale
          const float* cs = args.col_scale0 + static_cast<int64_t>(e) * args.ncols + nt * BN + c;
#pragma unroll
          for (int v = 0; v < 8; ++v) {
            const float4 u = __ldg(reinterpret_cast<const float4*>(cs + 4 * v));
            y[4 * v] = __float_as_uint(__uint_as_float(y[4 * v]) * (rs * u.x));
            y[4 * v + 1] = __float_as_uint(__uint_as_float(y[4 * v + 1]) * (rs * u.y));
            y[4 * v + 2] = __float_as_uint(__uint_as_float(y[4 * v + 2]) * (rs * u.z));
            y[4 * v + 3] = __float_as_uint(__uint_as_float(y[4 * v + 3]) * (rs * u.w));
          }
        }
        if (c > 0) {
          if (lane == 0) ptx::bulk_wait_group_read<0>();
          __syncwarp();
        }
        const uint32_t row = stg + lane * 128;
#pragma unroll
        for (int j = 0; j < 8; ++j)
          st_shared_v4(row + ((j ^ (lane & 7)) << 4), y[4 * j], y[4 * j + 1], y[4 * j + 2],
                       y[4 * j + 3]);
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          ptx::tma_store_2d(tmC, nt * BN + c, rbase, stg);
          ptx::bulk_commit_group();
        }
      }
      return;
    }
    // Stage the warp's 32 rows x 32 columns in shared memory, then store
    // them by row segments: lanes 8s..8s+7 write the 128 contiguous bytes
    // of one row, 4 rows per instruction (full lines, not one 16-byte
    // piece of 32 different rows).
    float* out0 = static_cast<float*>(args.out) + nt * BN;
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
      uint32_t y[32];
      ptx::tmem_ld32(tb + c, y);
      ptx::tmem_wait_ld();
      float4* mine = reinterpret_cast<float4*>(etile + lane * EPI_PITCH);
      if (FP8) {  // acc * row scale * channel scale
        const float* cs = args.col_scale0 + static_cast<int64_t>(e) * args.ncols + nt * BN + c;
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          const float4 u = __ldg(reinterpret_cast<const float4*>(cs + 4 * v));
          mine[v] = make_float4(__uint_as_float(y[4 * v]) * (rs * u.x),
                                __uint_as_float(y[4 * v + 1]) * (rs * u.y),
                                __uint_as_float(y[4 * v + 2]) * (rs * u.z),
                                __uint_as_float(y[4 * v + 3]) * (rs * u.w));
        }
      } else {
#pragma unroll
        for (int v = 0; v < 8; ++v)
          mine[v] = make_float4(__uint_as_float(y[4 * v]), __uint_as_float(y[4 * v + 1]),
                                __uint_as_float(y[4 * v + 2]), __uint_as_float(y[4 * v + 3]));
      }
      __syncwarp();
#pragma unroll
      for (int it = 0; it < 8; ++it) {
        const int r = it * 4 + sub;
        float4 val = *reinterpret_cast<const float4*>(etile + r * EPI_PITCH + col4);
        if (MODE == DGRAD_F32 && args.piece_cols > 0) {
          // piece_cols % 4 == 0: the 4 columns lie in one piece
          const int n = nt * BN + c + col4;
          const int pc = n / args.piece_cols;
          if (rbase + r < rend && pc < args.num_pieces)
            *reinterpret_cast<float4*>(static_cast<float*>(args.out) + pc * args.piece_stride +
                                       static_cast<int64_t>(rbase + r) * args.piece_cols + n -
                                       pc * args.piece_cols) = val;
        } else if (rbase + r < rend) {
          float4* dst = reinterpret_cast<float4*>(out0 + static_cast<int64_t>(rbase + r) * args.ldo +
                                                  c + col4);
          if (MODE == DGRAD_F32 && args.accumulate) {
            const float4 o = *dst;
            val = make_float4(o.x + val.x, o.y + val.y, o.z + val.z, o.w + val.w);
          }
          *dst = val;
        }
      }
      __syncwarp();
    }
  }
}

template <int MODE, bool FP8>
__global__ void __launch_bounds__(one_sm_threads<MODE, FP8>(), 1)
    tc_grouped_kernel(const __grid_constant__ CUtensorMap tmA,
                      const __grid_constant__ CUtensorMap tmB0,
                      const __grid_constant__ CUtensorMap tmB1,
                      const __grid_constant__ CUtensorMap tmC, TcArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* stages = smem;
  float* epi = reinterpret_cast<float*>(smem + STAGES * STAGE_BYTES);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES + EPI_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NUM_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* off = reinterpret_cast<int*>(tmem_slot + 4);
  int* tstart = off + (MOE_MAX_EXPERTS + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int E = args.E;
  const int NT = args.num_n_tiles;
  const int KB = args.k_blocks;
  const Ctl ctl{bars, abort_flag, args.err};

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(ctl.full(s), 1);
      ptx::mbar_init(ctl.empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(ctl.acc_full(b), 1);
      ptx::mbar_init(ctl.acc_empty(b), epi_warps<MODE, FP8>());
    }
    ptx::mbar_init(ctl.drain(), 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
    ptx::prefetch_tensormap(&tmA);
    ptx::prefetch_tensormap(&tmB0);
    ptx::prefetch_tensormap(&tmB1);
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), TMEM_COLS);
    ptx::tmem_relinquish();
  }
  load_offsets(off, args);
  __syncthreads();
  if (warp == 0) build_tile_prefix<BM>(off, tstart, E, NT, args.max_rows, args.err, lane);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total = tstart[E];

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      int stage = 0;
      uint32_t phase = 0;
      uint32_t fill_parity = 0, filled = 0;  // per stage: parity of its last fill
      bool alive = true;
      for (int tile = blockIdx.x; alive && tile < total; tile += gridDim.x) {
        int e, m0, rend, nt;
        decode_tile(tile, tstart, off, E, NT, e, m0, rend, nt);
        for (int kb = 0; kb < KB; ++kb) {
          if (!ctl.wait(ctl.empty(stage), phase ^ 1u, 1)) {
            alive = false;
            break;
          }
          const uint32_t fb = ctl.full(stage);
          ptx::mbar_arrive_expect_tx(fb, STAGE_BYTES);
          const uint32_t a = ptx::smem_u32(stages + stage * STAGE_BYTES);
          const uint32_t b = a + A_BYTES;
          int kc = kb * (FP8 ? KE_FP8 : BK);
          int arow = m0, eb = e;
          if (MODE == DGRAD_F32 && args.ksplit) {  // K split e of the dense rows
            arow = m0 - off[e];
            kc += e * KB * BK;
            eb = 0;
          }
          ptx::tma_load_2d(a, &tmA, kc, arow, fb);
          if (FP8) {
            // K-major weight rows: two boxes of 128 output channels x 128 K
            const int n0 = MODE == FC1 ? nt * (BN / 2) : nt * BN;
            ptx::tma_load_3d(b, &tmB0, kc, n0, e, fb);
            if (MODE == FC1)
              ptx::tma_load_3d(b + 2 * BOX_BYTES, &tmB1, kc, n0, e, fb);
            else
              ptx::tma_load_3d(b + 2 * BOX_BYTES, &tmB0, kc, n0 + BN / 2, e, fb);
          } else if (MODE == FC1 || MODE == FC1_BWD) {
            const int n0 = nt * (BN / 2);
            ptx::tma_load_3d(b, &tmB0, n0, kc, e, fb);
            ptx::tma_load_3d(b + BOX_BYTES, &tmB0, n0 + 64, kc, e, fb);
            ptx::tma_load_3d(b + 2 * BOX_BYTES, &tmB1, n0, kc, e, fb);
            ptx::tma_load_3d(b + 3 * BOX_BYTES, &tmB1, n0 + 64, kc, e, fb);
          } else if (MODE == DGRAD_BF16 || MODE == DGRAD_F32) {
            // K-major weight rows: two boxes of 128 output columns x 64 K
            const bool first = MODE == DGRAD_BF16 || kb < args.kb_split;
            const CUtensorMap* m = first ? &tmB0 : &tmB1;
            const int k1 = first ? kc : kc - args.kb_split * BK;
            ptx::tma_load_3d(b, m, k1, nt * BN, eb, fb);
            ptx::tma_load_3d(b + 2 * BOX_BYTES, m, k1, nt * BN + BN / 2, eb, fb);
          } else {
            const int n0 = nt * BN;
#pragma unroll
            for (int q = 0; q < 4; ++q) ptx::tma_load_3d(b + q * BOX_BYTES, &tmB0, n0 + 64 * q, kc, e, fb);
          }
          filled |= 1u << stage;
          fill_parity = (fill_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (alive) {
        // every filled stage released by the MMA warp: its commit-arrivals
        // have landed and no copy is in flight
        for (int i = 0; i < STAGES; ++i) {
          if (!ctl.wait(ctl.empty(stage), phase ^ 1u, 2, false)) break;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      } else {
        // give up: only wait (bounded) for the copies this thread issued
        for (int s = 0; s < STAGES; ++s)
          if (filled >> s & 1u) ctl.wait(ctl.full(s), fill_parity >> s & 1u, 3, false);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuer
      int stage = 0;
      uint32_t phase = 0;
      bool alive = true;
      int it = 0;
      for (int tile = blockIdx.x; alive && tile < total; tile += gridDim.x, ++it) {
        const int buf = it & 1;
        const uint32_t aph = (it >> 1) & 1;
        if (!ctl.wait(ctl.acc_empty(buf), aph ^ 1u, 4)) {
          alive = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d = tmem_base + buf * ACC_COLS;
        for (int kb = 0; kb < KB; ++kb) {
          if (!ctl.wait(ctl.full(stage), phase, 5)) {
            alive = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t a = ptx::smem_u32(stages + stage * STAGE_BYTES);
          const uint32_t b = a + A_BYTES;
          if (FP8) {
            // A and B both K-major, 128-byte swizzled rows, 8-row groups 1 KB
            // apart; a K step of 32 E4M3 values moves 32 B inside the row.
#pragma unroll
            for (int s = 0; s < KE_FP8 / 32; ++s) {
              const uint64_t adesc = ptx::smem_desc(a + s * 32, 16, 1024, ptx::kLayoutSw128);
              const uint64_t bdesc = ptx::smem_desc(b + s * 32, 16, 1024, ptx::kLayoutSw128);
              ptx::umma_e4m3(d, adesc, bdesc, IDESC_F8, (kb | s) != 0 ? 1u : 0u);
            }
          } else if (MODE == DGRAD_BF16 || MODE == DGRAD_F32) {
            // B K-major like A: 128-byte rows, 8-row groups 1 KB apart
#pragma unroll
            for (int s = 0; s < BK / 16; ++s) {
              const uint64_t adesc = ptx::smem_desc(a + s * 32, 16, A_SBO, A_LAYOUT);
              const uint64_t bdesc = ptx::smem_desc(b + s * 32, 16, 1024, ptx::kLayoutSw128);
              ptx::umma_bf16(d, adesc, bdesc, IDESC_KB, (kb | s) != 0 ? 1u : 0u);
            }
          } else {
#pragma unroll
          for (int s = 0; s < BK / 16; ++s) {
            // A: K-major, rows of BK bf16 (64 or 128 bytes) with the matching
            //    swizzle, 8-row groups A_SBO apart; a K step of 16 bf16 moves
            //    32 B inside the swizzled row.
            // B: MN-major, 128-byte swizzle; 64-column chunks (boxes)
            //    BOX_BYTES apart (LBO), 8-row K groups 1024 B apart (SBO); a K
            //    step of 16 rows moves 2048 B.
            const uint64_t adesc = ptx::smem_desc(a + s * 32, 16, A_SBO, A_LAYOUT);
            const uint64_t bdesc = ptx::sw128_desc(b + s * 2048, BOX_BYTES, 1024);
            ptx::umma_bf16(d, adesc, bdesc, IDESC, (kb | s) != 0 ? 1u : 0u);
          }
          }
          ptx::umma_commit(ctl.empty(stage));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!alive) break;
        ptx::umma_commit(ctl.acc_full(buf));
      }
      if (!alive) {
        ptx::umma_commit(ctl.drain());
        ctl.wait(ctl.drain(), 0, 6, false);
      }
    }
  } else {
    // ------------------------------------------------ epilogue warps 2..5 (2..9: E4M3 fc1)
    const int q = warp & 3;  // TMEM lane quarter this warp may read
    const int ch = epi_warps<MODE, FP8>() == 8 ? (warp - 2) / 4 : -1;  // its column half
    int it = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++it) {
      const int buf = it & 1;
      const uint32_t aph = (it >> 1) & 1;
      int e, m0, rend, nt;
      decode_tile(tile, tstart, off, E, NT, e, m0, rend, nt);
      bool ok = ctl.wait(ctl.acc_full(buf), aph, 7);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      ptx::tc_fence_after();
      const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * ACC_COLS;
      float* etile = epi + q * (EPI_WARP_BYTES / 4);  // this warp's staging region
      const uint32_t stg = ptx::smem_u32(etile);
      const int rbase = m0 + q * 32;  // this warp's first row; lane l holds row rbase + l
      drain_accumulator<MODE, FP8>(tb, etile, stg, &tmC, rbase, rend, nt, e, args, lane, ch);
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(ctl.acc_empty(buf));
    }
    if (args.tma_out && lane == 0) ptx::bulk_wait_group_all();  // the stores have completed
  }
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ------------------------------------------------------------------ SM pairs
// The same grouped GEMM on pairs of SMs: a 2-CTA cluster shares each MMA
// (tcgen05 cta_group::2).  One M=256,N=256,K=16 MMA covers 256 rows; the
// A rows are split 128/128 between the two CTAs' shared memories and so are
// the 256 B columns, so each SM stages half of the weight tile it multiplies
// by (half the shared-memory and L2 traffic per MMA of the one-SM kernel).
// A stage is then 32 KB per CTA (A 128x64, B 64x128), which leaves room for
// a 6-deep ring instead of 4.
//  * fc1 (and its backward recompute): rank 0 stages 128 columns of W1,
//    rank 1 the same 128 columns of W3, so accumulator column j and 128+j
//    are again the SwiGLU pair; fc2: rank r stages W2 columns
//    nt*256 + 128r .. +127; the dgrad modes: rank r stages the K-major rows
//    nt*256 + 128r .. +127 of the weight (one 128 x 64 box).
//  * Both CTAs' producers load their own halves; the copies of both count on
//    rank 0's full barrier (armed by rank 0 with both halves' bytes).  Rank 0
//    issues the MMAs; its commits arrive on the empty/acc_full barriers of
//    both CTAs.  Each CTA's TMEM holds the accumulator rows of its A half,
//    and its epilogue warps drain them and arrive on rank 0's acc_empty.
//  * A timed-out wait also raises the other CTA's abort flag, so the pair
//    gives up together; every cross-CTA access happens before the final
//    cluster barrier.
constexpr int PM = 2 * BM;                      // rows per pair tile
constexpr int P_STAGE_BYTES = A_BYTES + 2 * BOX_BYTES;
constexpr int P_STAGES = (SMEM_BUDGET - 1024 - EPI_BYTES - 4096) / P_STAGE_BYTES;  // 6 (BK=64)
constexpr int P_NUM_BARS = 2 * P_STAGES + 5;
constexpr int P_SMEM_BYTES = 1024 + P_STAGES * P_STAGE_BYTES + EPI_BYTES + P_NUM_BARS * 8 + 16 +
                             2 * (MOE_MAX_EXPERTS + 1) * 4;
static_assert(P_SMEM_BYTES <= SMEM_BUDGET, "shared memory budget (pair)");
static_assert(P_STAGES <= 32, "stage bit masks");
constexpr uint32_t P_IDESC = ptx::idesc_bf16_f32(PM, BN, /*b_mn_major=*/true);
constexpr uint32_t P_IDESC_F8 = ptx::idesc_e4m3_f32(PM, BN);
constexpr uint32_t P_IDESC_KB = ptx::idesc_bf16_f32(PM, BN, /*b_mn_major=*/false);
// Bounded pause that lets a CTA's own in-flight copies land when it gives up
// (their completion is counted on the other CTA's barrier).
constexpr long long kPeerDrainCycles = 20000000LL;
using PairCtl = CtlN<P_STAGES>;

template <int MODE, bool FP8>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
    tc_grouped_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                           const __grid_constant__ CUtensorMap tmB0,
                           const __grid_constant__ CUtensorMap tmB1,
                           const __grid_constant__ CUtensorMap tmC, TcArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* stages = smem;
  float* epi = reinterpret_cast<float*>(smem + P_STAGES * P_STAGE_BYTES);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + P_STAGES * P_STAGE_BYTES + EPI_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + P_NUM_BARS);
  int* abort_word = reinterpret_cast<int*>(tmem_slot + 1);
  volatile int* abort_flag = abort_word;
  int* off = reinterpret_cast<int*>(tmem_slot + 4);
  int* tstart = off + (MOE_MAX_EXPERTS + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();
  const int pair = blockIdx.x >> 1;
  const int npairs = gridDim.x >> 1;
  const int E = args.E;
  const int NT = args.num_n_tiles;
  const int KB = args.k_blocks;
  const PairCtl ctl{bars, abort_flag, args.err,
                    ptx::mapa_shared(ptx::smem_u32(abort_word), rank ^ 1u)};

  if (threadIdx.x == 0) {
    for (int s = 0; s < P_STAGES; ++s) {
      ptx::mbar_init(ctl.full(s), 1);
      ptx::mbar_init(ctl.empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(ctl.acc_full(b), 1);
      ptx::mbar_init(ctl.acc_empty(b), 8);  // 4 epilogue warps in each CTA
    }
    ptx::mbar_init(ctl.drain(), 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
    ptx::prefetch_tensormap(&tmA);
    ptx::prefetch_tensormap(&tmB0);
    ptx::prefetch_tensormap(&tmB1);
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(ptx::smem_u32(tmem_slot), TMEM_COLS);
    ptx::tmem_relinquish_pair();
  }
  load_offsets(off, args);
  __syncthreads();
  if (warp == 0) build_tile_prefix<PM>(off, tstart, E, NT, args.max_rows, args.err, lane);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();  // both CTAs' barriers initialised before any cross-CTA signal
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total = tstart[E];

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer (both CTAs)
      int stage = 0;
      uint32_t phase = 0;
      uint32_t fill_parity = 0, filled = 0;
      bool alive = true;
      // FC1 and its backward: rank 0 holds W1's 128 columns, rank 1 W3's
      constexpr bool kGate = MODE == FC1 || MODE == FC1_BWD;
      constexpr bool kDgrad = MODE == DGRAD_BF16 || MODE == DGRAD_F32;
      const CUtensorMap* tmB = (kGate && rank == 1) ? &tmB1 : &tmB0;
      for (int tile = pair; alive && tile < total; tile += npairs) {
        int e, m0, rend, nt;
        decode_tile<PM>(tile, tstart, off, E, NT, e, m0, rend, nt);
        const int n0 = kGate ? nt * (BN / 2) : nt * BN + static_cast<int>(rank) * (BN / 2);
        const int a_row = m0 + static_cast<int>(rank) * BM;
        for (int kb = 0; kb < KB; ++kb) {
          if (!ctl.wait(ctl.empty(stage), phase ^ 1u, 1)) {
            alive = false;
            break;
          }
          if (rank == 0) ptx::mbar_arrive_expect_tx(ctl.full(stage), 2 * P_STAGE_BYTES);
          const uint32_t fb = ptx::mapa_shared(ctl.full(stage), 0);
          const uint32_t a = ptx::smem_u32(stages + stage * P_STAGE_BYTES);
          const uint32_t b = a + A_BYTES;
          int kc = kb * (FP8 ? KE_FP8 : BK);
          int arow = a_row, eb = e;
          if (MODE == DGRAD_F32 && args.ksplit) {  // K split e of the dense rows
            arow = a_row - off[e];
            kc += e * KB * BK;
            eb = 0;
          }
          ptx::tma_load_2d_pair(a, &tmA, kc, arow, fb);
          if (FP8) {
            // K-major weight rows: one box of this CTA's 128 output channels x 128 K
            ptx::tma_load_3d_pair(b, tmB, kc, n0, e, fb);
          } else if (kDgrad) {
            // K-major weight rows: one box of this CTA's 128 output columns x
            // 64 K, from the weight that holds this K block
            const bool first = MODE == DGRAD_BF16 || kb < args.kb_split;
            ptx::tma_load_3d_pair(b, first ? &tmB0 : &tmB1, first ? kc : kc - args.kb_split * BK,
                                  n0, eb, fb);
          } else {
            ptx::tma_load_3d_pair(b, tmB, n0, kc, e, fb);
            ptx::tma_load_3d_pair(b + BOX_BYTES, tmB, n0 + 64, kc, e, fb);
          }
          filled |= 1u << stage;
          fill_parity = (fill_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == P_STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (alive) {
        // every filled stage released by the MMAs (the commits arrive in both CTAs)
        for (int i = 0; i < P_STAGES; ++i) {
          if (!ctl.wait(ctl.empty(stage), phase ^ 1u, 2, false)) break;
          if (++stage == P_STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      } else if (rank == 0) {
        for (int s = 0; s < P_STAGES; ++s)
          if (filled >> s & 1u) ctl.wait(ctl.full(s), fill_parity >> s & 1u, 3, false);
      } else {
        const long long t0 = clock64();
        while (clock64() - t0 < kPeerDrainCycles) {
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ------------------------------------------------ MMA issuer (rank 0)
      int stage = 0;
      uint32_t phase = 0;
      bool alive = true;
      int it = 0;
      for (int tile = pair; alive && tile < total; tile += npairs, ++it) {
        const int buf = it & 1;
        const uint32_t aph = (it >> 1) & 1;
        if (!ctl.wait(ctl.acc_empty(buf), aph ^ 1u, 4)) {
          alive = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d = tmem_base + buf * ACC_COLS;
        for (int kb = 0; kb < KB; ++kb) {
          if (!ctl.wait(ctl.full(stage), phase, 5)) {
            alive = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t a = ptx::smem_u32(stages + stage * P_STAGE_BYTES);
          const uint32_t b = a + A_BYTES;
          if (FP8) {
            // both operands K-major (128-byte rows), K = 32 per MMA
#pragma unroll
            for (int s = 0; s < KE_FP8 / 32; ++s) {
              const uint64_t adesc = ptx::smem_desc(a + s * 32, 16, 1024, ptx::kLayoutSw128);
              const uint64_t bdesc = ptx::smem_desc(b + s * 32, 16, 1024, ptx::kLayoutSw128);
              ptx::umma_e4m3_pair(d, adesc, bdesc, P_IDESC_F8, (kb | s) != 0 ? 1u : 0u);
            }
          } else if (MODE == DGRAD_BF16 || MODE == DGRAD_F32) {
            // B K-major like A in each CTA: 128 rows of 128 bytes, 8-row
            // groups 1 KB apart
#pragma unroll
            for (int s = 0; s < BK / 16; ++s) {
              const uint64_t adesc = ptx::smem_desc(a + s * 32, 16, A_SBO, A_LAYOUT);
              const uint64_t bdesc = ptx::smem_desc(b + s * 32, 16, 1024, ptx::kLayoutSw128);
              ptx::umma_bf16_pair(d, adesc, bdesc, P_IDESC_KB, (kb | s) != 0 ? 1u : 0u);
            }
          } else {
#pragma unroll
            for (int s = 0; s < BK / 16; ++s) {
              // same descriptors as the one-SM kernel, read at the same
              // offsets in both CTAs' shared memories; B has two 64-column
              // boxes per CTA
              const uint64_t adesc = ptx::smem_desc(a + s * 32, 16, A_SBO, A_LAYOUT);
              const uint64_t bdesc = ptx::sw128_desc(b + s * 2048, BOX_BYTES, 1024);
              ptx::umma_bf16_pair(d, adesc, bdesc, P_IDESC, (kb | s) != 0 ? 1u : 0u);
            }
          }
          ptx::umma_commit_pair(ctl.empty(stage), 3);
          if (++stage == P_STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!alive) break;
        ptx::umma_commit_pair(ctl.acc_full(buf), 3);
      }
      if (!alive) {
        ptx::umma_commit_pair(ctl.drain(), 1);
        ctl.wait(ctl.drain(), 0, 6, false);
      }
    }
  } else {
    // ------------------------------------------------ epilogue warps 2..5 (both CTAs)
    const int q = warp & 3;
    int it = 0;
    for (int tile = pair; tile < total; tile += npairs, ++it) {
      const int buf = it & 1;
      const uint32_t aph = (it >> 1) & 1;
      int e, m0, rend, nt;
      decode_tile<PM>(tile, tstart, off, E, NT, e, m0, rend, nt);
      bool ok = ctl.wait(ctl.acc_full(buf), aph, 7);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      ptx::tc_fence_after();
      const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * ACC_COLS;
      float* etile = epi + q * (EPI_WARP_BYTES / 4);
      const uint32_t stg = ptx::smem_u32(etile);
      const int rbase = m0 + static_cast<int>(rank) * BM + q * 32;
      drain_accumulator<MODE, FP8>(tb, etile, stg, &tmC, rbase, rend, nt, e, args, lane);
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_cluster(ptx::mapa_shared(ctl.acc_empty(buf), 0));
    }
    if (args.tma_out && lane == 0) ptx::bulk_wait_group_all();  // the stores have completed
  }
  __syncthreads();
  ptx::cluster_sync();  // no cross-CTA access after this point
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

// ------------------------------------------------------------------ host side
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

// 2-D bf16 activation map [rows, inner], box BK (inner) x 128 (rows), with the
// swizzle whose span equals the box's row (64 or 128 bytes).
bool map_rows(CUtensorMap* m, const void* ptr, int64_t inner, int64_t rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(inner) * 2};
  cuuint32_t box[2] = {BK, BM};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE,
             BK == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D bf16 weight map [E, K, N] (N contiguous), box 64 (N) x BK (K) x 1.
bool map_weights(CUtensorMap* m, const void* ptr, int64_t N, int64_t K, int64_t E) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(K),
                        static_cast<cuuint64_t>(E)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(N) * 2, static_cast<cuuint64_t>(N * K) * 2};
  cuuint32_t box[3] = {64, BK, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// E4M3 maps: activations [rows, K] bytes, box 128 (K) x 128 (rows); K-major
// weights [E, N, K] bytes, box 128 (K) x 128 (N) x 1; both 128-byte swizzle.
bool map_rows_e4m3(CUtensorMap* m, const void* ptr, int64_t K, int64_t rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(K)};
  cuuint32_t box[2] = {KE_FP8, BM};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
bool map_weights_e4m3(CUtensorMap* m, const void* ptr, int64_t K, int64_t N, int64_t E) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(N),
                        static_cast<cuuint64_t>(E)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(N * K)};
  cuuint32_t box[3] = {KE_FP8, 128, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(ptr), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// bf16 K-major weight view [E, N, K] of a weight stored [E][N][K] (K
// contiguous), box 64 (K) x 128 (N) x 1, 128-byte swizzle: W2 [E, f, h] seen
// with K = h for fc2's dgrad, W1/W3 [E, h, f] with K = f for fc1's.
bool map_weights_kmajor(CUtensorMap* m, const void* ptr, int64_t K, int64_t N, int64_t E) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(N),
                        static_cast<cuuint64_t>(E)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(K) * 2, static_cast<cuuint64_t>(N * K) * 2};
  cuuint32_t box[3] = {64, 128, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp32 output [rows, N] with row stride ld floats, box 32 (N) x 32 (rows),
// 128-byte swizzle: the epilogue's TMA stores.  False when the layout cannot
// be stored by TMA (stride or base not 16-byte aligned).
bool map_out_f32(CUtensorMap* m, float* ptr, int64_t N, int64_t ld, int64_t rows) {
  if (ld % 4 != 0 || (reinterpret_cast<uintptr_t>(ptr) & 15) != 0 || N % 32 != 0) return false;
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 4};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, ptr, dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D fp16 output map [rows, N] (row stride ld elements), box 64 x 32 in the
// 128-byte swizzle: one epilogue warp's 32 rows x 64 columns per store.
bool map_out_f16(CUtensorMap* m, void* ptr, int64_t N, int64_t ld, int64_t rows) {
  if (ld % 8 != 0 || (reinterpret_cast<uintptr_t>(ptr) & 15) != 0 || N % 64 != 0) return false;
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
  cuuint32_t box[2] = {64, 32};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, ptr, dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Sets args->tma_out and fills *c when the fp32 output [max_rows, N] (row
// stride args->ldo) can be stored by TMA; MOE_TC_TMA_OUT=0 in the
// environment keeps the row-segment stores (a tuning override).
void setup_tma_out(CUtensorMap* c, TcArgs* args, int64_t N) {
  const char* force = getenv("MOE_TC_TMA_OUT");
  if (force && force[0] == '0') return;
  if (args->accumulate) return;
  if (map_out_f32(c, static_cast<float*>(args->out), N, args->ldo, args->max_rows))
    args->tma_out = 1;
}

template <int MODE, bool FP8>
cudaError_t launch_tc(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1,
                      const CUtensorMap& c, const TcArgs& args, cudaStream_t s) {
  static bool configured[64] = {false};
  int dev = 0;
  cudaError_t st = cudaGetDevice(&dev);
  if (st != cudaSuccess) return st;
  if (dev < 64 && !configured[dev]) {
    st = cudaFuncSetAttribute(tc_grouped_kernel<MODE, FP8>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (st != cudaSuccess) return st;
    configured[dev] = true;
  }
  const int64_t max_tiles = ((args.max_rows + BM - 1) / BM + args.E) * args.num_n_tiles;
  int64_t grid = device_sm_count();
  if (grid > max_tiles) grid = max_tiles;
  if (grid <= 0) return cudaSuccess;
  tc_grouped_kernel<MODE, FP8><<<static_cast<unsigned>(grid), one_sm_threads<MODE, FP8>(),
                                 SMEM_BYTES, s>>>(a, b0, b1, c, args);
  return cudaGetLastError();
}

// Pairs of SMs that can be resident at once for the pair kernel (0: none, or
// the query failed).
template <int MODE, bool FP8>
int pair_slots() {
  static int cache[64] = {0};  // per device; -1 = queried, unusable
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (cache[dev] == 0) {
    int n = 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = P_SMEM_BYTES;
    if (cudaFuncSetAttribute(tc_grouped_pair_kernel<MODE, FP8>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             P_SMEM_BYTES) != cudaSuccess ||
        cudaOccupancyMaxActiveClusters(&n, tc_grouped_pair_kernel<MODE, FP8>, &cfg) !=
            cudaSuccess ||
        n <= 0) {
      cudaGetLastError();  // clear a failed query; the one-SM kernel is used instead
      n = -1;
    }
    cache[dev] = n;
  }
  return cache[dev] > 0 ? cache[dev] : 0;
}

template <int MODE, bool FP8>
cudaError_t launch_tc_pair(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1,
                           const CUtensorMap& c, const TcArgs& args, int slots, cudaStream_t s) {
  const int64_t max_tiles = ((args.max_rows + PM - 1) / PM + args.E) * args.num_n_tiles;
  int64_t pairs = slots;
  if (pairs > max_tiles) pairs = max_tiles;
  if (pairs <= 0) return cudaSuccess;
  tc_grouped_pair_kernel<MODE, FP8><<<static_cast<unsigned>(2 * pairs), THREADS, P_SMEM_BYTES, s>>>(
      a, b0, b1, c, args);
  return cudaGetLastError();
}

// Experts averaging at least this many rows run on SM pairs (256-row tiles);
// fewer rows per expert keep 128-row tiles on single SMs, where a 256-row
// tile would mostly compute rows that are not stored.  MOE_TC_PAIR=0 / =1 in
// the environment forces one kernel or the other (a tuning override).
constexpr int64_t kPairMinRows = 768;

template <int MODE, bool FP8>
cudaError_t launch_grouped(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1,
                           const CUtensorMap& c, const TcArgs& args, cudaStream_t s) {
  const char* force = getenv("MOE_TC_PAIR");
  bool pair = args.max_rows >= static_cast<int64_t>(args.E) * kPairMinRows;
  if (force && force[0] == '0') pair = false;
  if (force && force[0] == '1') pair = true;
  if (pair) {
    const int slots = pair_slots<MODE, FP8>();
    if (slots > 0) return launch_tc_pair<MODE, FP8>(a, b0, b1, c, args, slots, s);
  }
  return launch_tc<MODE, FP8>(a, b0, b1, c, args, s);
}

}  // namespace

cudaError_t launch_tc_fc1(int E, int h, int f, int64_t max_rows, const void* x_perm,
                          const int32_t* offsets, const void* W1, const void* W3, void* h_mid,
                          int* err, cudaStream_t s) {
  if (max_rows == 0) return cudaSuccess;
  CUtensorMap a, b0, b1;
  if (!map_rows(&a, x_perm, h, max_rows) || !map_weights(&b0, W1, f, h, E) ||
      !map_weights(&b1, W3, f, h, E))
    return cudaErrorInvalidValue;
  TcArgs args{offsets, E, f / (BN / 2), h / BK, max_rows, h_mid, f, err};
  return launch_grouped<FC1, false>(a, b0, b1, a, args, s);
}

cudaError_t launch_tc_fc2(int E, int h, int f, int64_t max_rows, const void* h_mid,
                          const int32_t* offsets, const void* W2, float* y_perm, int* err,
                          cudaStream_t s) {
  if (max_rows == 0) return cudaSuccess;
  CUtensorMap a, b0;
  if (!map_rows(&a, h_mid, f, max_rows) || !map_weights(&b0, W2, h, f, E))
    return cudaErrorInvalidValue;
  TcArgs args{offsets, E, h / BN, f / BK, max_rows, y_perm, h, err};
  CUtensorMap c = a;
  setup_tma_out(&c, &args, h);
  return launch_grouped<FC2, false>(a, b0, b0, c, args, s);
}

cudaError_t launch_tc_fc2_top1(int E, int h, int f, int64_t max_rows, const void* h_mid,
                               const int32_t* offsets, const void* W2, const int32_t* row_token,
                               const float* row_weight, void* y, int* err, cudaStream_t s) {
  if (max_rows == 0) return cudaSuccess;
  CUtensorMap a, b0;
  if (!map_rows(&a, h_mid, f, max_rows) || !map_weights(&b0, W2, h, f, E))
    return cudaErrorInvalidValue;
  TcArgs args{offsets, E, h / BN, f / BK, max_rows, y, h, err};
  args.row_token = row_token;
  args.row_weight = row_weight;
  return launch_grouped<FC2_Y, false>(a, b0, b0, a, args, s);
}

cudaError_t launch_tc_fc2_f16s(int E, int h, int f, int64_t max_rows, const void* h_mid,
                               const int32_t* offsets, const void* W2, void* y16, int8_t* y16_exp,
                               int* err, cudaStream_t s) {
  if (max_rows == 0) return cudaSuccess;
  CUtensorMap a, b0;
  if (!map_rows(&a, h_mid, f, max_rows) || !map_weights(&b0, W2, h, f, E))
    return cudaErrorInvalidValue;
  TcArgs args{offsets, E, h / BN, f / BK, max_rows, y16, h, err};
  args.exp_out = y16_exp;
  CUtensorMap c = a;  // whole warps store by TMA (MOE_TC_TMA_OUT=0 keeps per-lane stores)
  const char* force = getenv("MOE_TC_TMA_OUT");
  if (!(force && force[0] == '0') && map_out_f16(&c, y16, h, h, max_rows)) args.tma_out = 1;
  return launch_grouped<FC2_F16S, false>(a, b0, b0, c, args, s);
}

// ---- backward GEMMs (bf16 operands, 64-wide K stages; SM pairs by the
// forward's rule)

cudaError_t launch_tc_dgrad_fc2(int E, int h, int f, int64_t max_rows, const void* dY,
                                const int32_t* offsets, const void* W2, void* dH, int* err,
                                cudaStream_t s) {
  if (BK != 64) return cudaErrorNotSupported;
  if (max_rows == 0) return cudaSuccess;
  CUtensorMap a, b0;
  if (!map_rows(&a, dY, h, max_rows) || !map_weights_kmajor(&b0, W2, h, f, E))
    return cudaErrorInvalidValue;
  // f % 128 == 0: the last 256-column tile may hold only 128 valid columns
  TcArgs args{offsets, E, (f + BN - 1) / BN, h / BK, max_rows, dH, f, err};
  args.ncols = f;
  return launch_grouped<DGRAD_BF16, false>(a, b0, b0, a, args, s);
}

cudaError_t launch_tc_fc1_bwd(int E, int h, int f, int64_t max_rows, const void* x_perm,
                              const int32_t* offsets, const void* W1, const void* W3,
                              const void* dH, void* dA, int* err, cudaStream_t s) {
  if (BK != 64) return cudaErrorNotSupported;
  if (max_rows == 0) return cudaSuccess;
  CUtensorMap a, b0, b1;
  if (!map_rows(&a, x_perm, h, max_rows) || !map_weights(&b0, W1, f, h, E) ||
      !map_weights(&b1, W3, f, h, E))
    return cudaErrorInvalidValue;
  TcArgs args{offsets, E, f / (BN / 2), h / BK, max_rows, dA, 2 * f, err};
  args.aux = dH;
  args.ldaux = f;
  args.ncols = f;
  return launch_grouped<FC1_BWD, false>(a, b0, b1, a, args, s);
}

cudaError_t launch_tc_dgrad_fc1(int E, int h, int f, int64_t max_rows, const void* dA,
                                const int32_t* offsets, const void* W1, const void* W3,
                                float* dX, int* err, cudaStream_t s, bool accumulate) {
  if (BK != 64) return cudaErrorNotSupported;
  if (max_rows == 0) return cudaSuccess;
  CUtensorMap a, b0, b1;
  if (!map_rows(&a, dA, 2 * f, max_rows) || !map_weights_kmajor(&b0, W1, f, h, E) ||
      !map_weights_kmajor(&b1, W3, f, h, E))
    return cudaErrorInvalidValue;
  TcArgs args{offsets, E, h / BN, 2 * f / BK, max_rows, dX, h, err};
  args.kb_split = f / BK;
  args.accumulate = accumulate ? 1 : 0;
  CUtensorMap c = a;
  setup_tma_out(&c, &args, h);
  return launch_grouped<DGRAD_F32, false>(a, b0, b1, c, args, s);
}

// C [rows, N] fp32 (row stride ldc) = A [rows, K] . Bk [N, K]^T, bf16
// operands, one dense group (the DGRAD_F32 mainloop with every K block from
// Bk); K % 64 == 0, N % 256 == 0.  The router's dx = dl . Wg^T runs here on
// bf16 hi/lo splits of its fp32 operands.
cudaError_t launch_tc_dense_nt_f32(int64_t rows, int K, int N, const void* A, const void* Bk,
                                   float* C, int ldc, int* err, cudaStream_t s) {
  if (BK != 64) return cudaErrorNotSupported;
  if (K % BK != 0 || N % BN != 0) return cudaErrorInvalidValue;
  if (rows == 0) return cudaSuccess;
  CUtensorMap a, b0;
  if (!map_rows(&a, A, K, rows) || !map_weights_kmajor(&b0, Bk, K, N, 1))
    return cudaErrorInvalidValue;
  TcArgs args{nullptr, 1, N / BN, K / BK, rows, C, ldc, err};
  args.kb_split = K / BK;
  CUtensorMap c = a;
  setup_tma_out(&c, &args, N);
  return launch_grouped<DGRAD_F32, false>(a, b0, b0, c, args, s);
}

int router_ksplit(int h) {
  const char* force = getenv("MOE_ROUTER_KSPLIT");  // a tuning override
  int S = (h + kRouterChainK - 1) / kRouterChainK;
  if (force && force[0] >= '1' && force[0] <= '9') S = force[0] - '0';
  if (S > kRouterMaxSplits / 3) S = kRouterMaxSplits / 3;
  const int kb = h / BK;
  if (S > kb) S = kb;
  return S < 1 ? 1 : S;
}

cudaError_t launch_tc_router_logits(int T, int h, int E, const void* x, const void* Wk,
                                    float* partials, int* nsplit, int* err, cudaStream_t s) {
  if (BK != 64) return cudaErrorNotSupported;
  if (h % BK != 0 || E % 4 != 0) return cudaErrorInvalidValue;
  const int S = router_ksplit(h);
  *nsplit = 3 * S;
  if (T == 0) return cudaSuccess;
  CUtensorMap a, b0;
  // B rows past the 3E of the pieces, and K past h (the last split's ragged
  // end), read as zeros; columns past 3E are not stored
  if (!map_rows(&a, x, h, T) || !map_weights_kmajor(&b0, Wk, h, 3 * E, 1))
    return cudaErrorInvalidValue;
  const int kbs = (h / BK + S - 1) / S;  // K blocks per split
  TcArgs args{nullptr, S, (3 * E + BN - 1) / BN, kbs, static_cast<int64_t>(S) * T, partials, E,
              err};
  args.kb_split = kbs;
  args.ksplit = 1;
  args.piece_cols = E;
  args.num_pieces = 3;
  args.piece_stride = static_cast<int64_t>(S) * T * E;  // partial (piece p, split e): p * S + e
  return launch_grouped<DGRAD_F32, false>(a, b0, b0, a, args, s);
}

cudaError_t launch_tc_fc1_e4m3(int E, int h, int f, int64_t max_rows, const uint8_t* xq,
                               const float* x_scale, const int32_t* row_src,
                               const int32_t* offsets, const uint8_t* W1q, const float* s1,
                               const uint8_t* W3q, const float* s3, void* h_mid, int* err,
                               cudaStream_t s) {
  if (max_rows == 0) return cudaSuccess;
  CUtensorMap a, b0, b1;
  if (!map_rows_e4m3(&a, xq, h, max_rows) || !map_weights_e4m3(&b0, W1q, h, f, E) ||
      !map_weights_e4m3(&b1, W3q, h, f, E))
    return cudaErrorInvalidValue;
  TcArgs args{offsets, E, f / (BN / 2), h / KE_FP8, max_rows, h_mid, f, err};
  args.row_scale = x_scale;
  args.row_src = row_src;
  args.col_scale0 = s1;
  args.col_scale1 = s3;
  args.ncols = f;
  return launch_grouped<FC1, true>(a, b0, b1, a, args, s);
}

cudaError_t launch_tc_fc2_e4m3_f16s(int E, int h, int f, int64_t max_rows, const uint8_t* hq,
                                    const float* h_scale, const int32_t* offsets,
                                    const uint8_t* W2q, const float* s2, void* y16,
                                    int8_t* y16_exp, int* err, cudaStream_t s) {
  if (max_rows == 0) return cudaSuccess;
  CUtensorMap a, b0;
  if (!map_rows_e4m3(&a, hq, f, max_rows) || !map_weights_e4m3(&b0, W2q, f, h, E))
    return cudaErrorInvalidValue;
  TcArgs args{offsets, E, h / BN, f / KE_FP8, max_rows, y16, h, err};
  args.row_scale = h_scale;
  args.col_scale0 = s2;
  args.ncols = h;
  args.exp_out = y16_exp;
  CUtensorMap c = a;
  const char* force = getenv("MOE_TC_TMA_OUT");
  if (!(force && force[0] == '0') && map_out_f16(&c, y16, h, h, max_rows)) args.tma_out = 1;
  return launch_grouped<FC2_F16S, true>(a, b0, b0, c, args, s);
}

cudaError_t launch_tc_fc2_e4m3(int E, int h, int f, int64_t max_rows, const uint8_t* hq,
                               const float* h_scale, const int32_t* offsets, const uint8_t* W2q,
                               const float* s2, float* y_perm, int* err, cudaStream_t s) {
  if (max_rows == 0) return cudaSuccess;
  CUtensorMap a, b0;
  if (!map_rows_e4m3(&a, hq, f, max_rows) || !map_weights_e4m3(&b0, W2q, f, h, E))
    return cudaErrorInvalidValue;
  TcArgs args{offsets, E, h / BN, f / KE_FP8, max_rows, y_perm, h, err};
  args.row_scale = h_scale;
  args.col_scale0 = s2;
  args.ncols = h;
  CUtensorMap c = a;
  setup_tma_out(&c, &args, h);
  return launch_grouped<FC2, true>(a, b0, b0, c, args, s);
}

}  // namespace moe
