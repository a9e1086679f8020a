// Block-scaled FP8 GEMM with per-128-K promotion into FP32 (sm_103a).
//
// Method (page 2, inprokorea.com free #735329): the tensor cores accumulate
// only within one K group; after each group of 128 the partial result is moved
// to FP32 registers on the CUDA cores, multiplied by the group's activation
// tile scale and weight block scale, and added to a full-precision FP32
// accumulator (promotion passage, Figure 6; per-group-scaling passage).  The
// pages describe this on H800 with two warpgroups alternating WGMMA and
// promotion (page 1, passage on two concurrent WGMMAs); that is prior art.
//
// B300 design (one persistent CTA per SM, 384 threads, 1 CTA/SM):
//   warp 8      TMA producer: one 128x128 A tile + one 256x128 B tile of E4M3
//               codes per 128-K slice into a 4-stage ring (128-byte swizzle).
//   warp 9      MMA issuer: one elected lane of the converged warp issues
//               4 x tcgen05.mma (M128 N256 K32, kind::f8f6f4, FP32 accumulate)
//               per slice into one of two TMEM buffers (2 x 256 columns), then
//               commits to the stage's "empty" barrier and the buffer's "full"
//               barrier.
//   warps 0-7   promotion/epilogue: warp w reads TMEM lanes 32(w%4).. (its 32
//               rows) and columns 128(w/4).. (its half of N) of the finished
//               buffer with tcgen05.ld, frees the buffer, and does
//               acc += P * (sa[row,kb] * sb[.,kb]) with packed f32x2 FMAs.
//               The FP32 accumulator (128 values per thread) stays in
//               registers for the whole tile; TMEM only ever holds one
//               slice's partial, so the MMA of slice kb+1 overlaps the
//               promotion of slice kb, and the next tile's MMAs overlap this
//               tile's final store.
// Output (dense): each promotion warp converts its 32 x 128 block chunk by
// chunk (32 rows x 64 bytes) into a 2 KB shared staging buffer laid out in the
// tensor map's 64-byte swizzle and writes it with one TMA tile store, which
// clips at the matrix bounds.  Per-thread row stores (16 bytes into 32
// different rows per instruction) take two to three times as long, and the
// tensor pipe idles meanwhile.  The grouped kernel does the same for warps
// whose rows lie inside one expert, and per-thread row stores, masked at the
// expert's end, for a warp that straddles it.
// Output modes (template EPI): EPI_STORE writes C in BF16 or FP32; EPI_QUANT
// (dense) quantises each thread's 128 columns of its row -- one 1x128 tile --
// with the activation quantiser's rules and stores codes through the same
// staging; EPI_SWIGLU (grouped) loads each B stage as gate/up/gate/up 64-row
// boxes so that a thread holds g and u of the same 64 outputs, forms
// h = silu(g) * u and stores h's codes and power-of-2 scales; EPI_WHOLEK is a
// study mode that accumulates all of K in TMEM with per-tensor scales.
// Tiles are visited in groups of M-tiles (all N-tiles of a group before the
// next), so a group's A rows stay in L2 while B streams once per group.  The
// host sizes a group to at most kGroupABytes of A (the Fprop shape, M = 4096 at
// K = 7168, is one group: B is read from DRAM once).
// Every pipeline wait is bounded (FP8FG_ERR_TIMEOUT, see device_common.cuh).

#include <cuda_bf16.h>

#include <cstddef>

#include "device_common.cuh"
#include "launch.h"

namespace fp8fg {

namespace {

constexpr int BM = 128, BN = 256, BK = 128;
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK;
constexpr int B_BYTES = BN * BK;
constexpr int NUM_EPI_WARPS = 8;
constexpr int PRODUCER_WARP = 8;
constexpr int MMA_WARP = 9;
constexpr int NUM_THREADS = 384;      // 3 warpgroups: 2 promotion/epilogue, 1 TMA+MMA
// Register split (per thread): launched at 168 (= 65536 / 384 rounded down to 8);
// the TMA/MMA warpgroup gives up to 56 and the two promotion warpgroups take 224:
// 2 x 224 + 56 = 3 x 168, so the re-allocation never waits on registers.
constexpr int REGS_LAUNCH = 168;
constexpr int REGS_PRODUCER = 56;
constexpr int REGS_EPILOGUE = 224;
static_assert(2 * REGS_EPILOGUE + REGS_PRODUCER <= 3 * REGS_LAUNCH, "register split");
// The grouped kernels spill at the 224/56 split (their TMA/MMA warpgroup needs
// more than 56 registers for the expert-tile lookup): the plain grouped kernel
// runs at 184/136 and the SwiGLU kernel at 208/88, both without spills.
constexpr int SWIGLU_REGS_EPILOGUE = 208;
constexpr int GROUPED_REGS_EPILOGUE = 184;
__host__ __device__ constexpr int regs_epilogue(bool grouped, int epi) {
  return epi == 2 ? SWIGLU_REGS_EPILOGUE : grouped ? GROUPED_REGS_EPILOGUE : REGS_EPILOGUE;
}
__host__ __device__ constexpr int regs_producer(bool grouped, int epi) {
  return (3 * REGS_LAUNCH - 2 * regs_epilogue(grouped, epi)) / 8 * 8;
}
static_assert(2 * SWIGLU_REGS_EPILOGUE + regs_producer(true, 2) <= 3 * REGS_LAUNCH, "register split");
static_assert(2 * GROUPED_REGS_EPILOGUE + regs_producer(true, 0) <= 3 * REGS_LAUNCH, "register split");
constexpr int TMEM_COLS = 512;
// A bytes one tile group may hold in L2 (126 MB): room is left for the B tiles
// in flight and the output's write-back.
constexpr int64_t kGroupABytes = int64_t{48} << 20;
constexpr int MAX_EXPERTS = 1024;
constexpr int SCALE_WARP = 10;        // tile mode: loads and transposes the B column scales
constexpr int SB = 4;                 // tile mode: slices per scale-ring slot
constexpr int SB_SLOTS = 2;           // tile mode: scale-ring slots
constexpr int CST_BYTES = 2048;       // output staging per promotion warp: 32 rows x 64 bytes
constexpr int CST_ROW = 64;           // bytes per staged row (the tensor map's 64-byte swizzle)
constexpr uint32_t IDESC = idesc_e4m3_f32(BM, BN);
// Output modes of the kernel's store phase.
constexpr int EPI_STORE = 0;    // C in BF16 or FP32
constexpr int EPI_QUANT = 1;    // dense: C as 1x128 E4M3 tiles + scales
constexpr int EPI_SWIGLU = 2;   // grouped: h = silu(gate) * up as 1x128 E4M3 tiles + scales
// Study mode (dense, block path): no per-slice promotion.  All of K accumulates
// in one TMEM buffer per tile and is scaled once by per-tensor scales
// sa[0] * sb[0]; this measures the tensor core's own FP8 accumulation.
constexpr int EPI_WHOLEK = 3;

struct GemmParams {
  const float* sa;        // [rows, nkb]
  const float* sb;        // block: [E][N/128][nkb]; tile: [N][nkb]
  void* c;                // [rows, N]
  const int32_t* offsets; // grouped only, [E+1]
  int M;                  // dense: rows of A/C; grouped: total rows
  int N, K, nkb;
  int m_tiles, n_tiles;   // dense tiling (m_tiles unused when grouped)
  int group_m;            // dense: M-tiles per tile group (see tile_of)
  int E;
  int c_f32;
  int b_tile;
  float* s_out;           // quantised output: [rows, N/128] tile scales
  int pow2_out;           // quantised output: power-of-2 scales
  long long wait_limit;
  int* status;            // library status word
  // Work split (see WorkList): tiles [0, dp_tiles) are whole tiles taken
  // round-robin; each of the sk_tiles tiles after them is shared by its own
  // group of CTAs, which divide its 128-K slices evenly (stream-K).  A tile
  // shared by several CTAs leaves FP32 partial sums in the workspace
  // ([sk_grid][BM][BN], one slot per CTA); the fix-up kernel adds them up.
  int dp_tiles = INT32_MAX;
  int sk_tiles = 0;
  int sk_grid = 0;        // CTAs taking part in the split (the fix-up recomputes it)
};

// One unit of a CTA's work: slices [kb0, kb1) of tile t.  slot -1: the whole
// tile (its result goes to C); 0: a part of a tile shared between CTAs, whose
// partial sum goes to the CTA's workspace slot.
struct Work {
  int t, kb0, kb1, slot;
};

// The stream-K group of CTAs sharing split tile j (R = sk_tiles <= G = sk_grid
// CTAs): CTAs [first(j), first(j + 1)) with first(j) = ceil(j G / R); CTA b
// belongs to tile floor(b R / G).
__host__ __device__ __forceinline__ int sk_first_cta(int j, int R, int G) {
  return static_cast<int>((static_cast<long long>(j) * G + R - 1) / R);
}
// Slices [kb0, kb1) of its tile that member i of a group of n CTAs takes.
__host__ __device__ __forceinline__ void sk_share(int i, int n, int nkb, int& kb0, int& kb1) {
  kb0 = static_cast<int>(static_cast<long long>(i) * nkb / n);
  kb1 = static_cast<int>(static_cast<long long>(i + 1) * nkb / n);
}

// The sequence of units of this CTA, the same for every warp role.  A launch
// without SK takes the whole tiles [0, dp_tiles) round-robin; the split launch
// of a dense GEMM that stores C (SK) takes only its CTA's share of one of the
// tiles after them.
template <bool SK>
struct WorkList {
  int next_dp;
  bool sk_pending;
  __device__ __forceinline__ void init(const GemmParams& p) {
    next_dp = SK ? INT32_MAX : static_cast<int>(blockIdx.x);
    sk_pending = SK && static_cast<int>(blockIdx.x) < p.sk_grid && p.sk_tiles > 0;
  }
  __device__ __forceinline__ bool next(const GemmParams& p, int num_tiles, Work& w) {
    if (next_dp < min(p.dp_tiles, num_tiles)) {
      w = {next_dp, 0, p.nkb, -1};
      next_dp += gridDim.x;
      return true;
    }
    if constexpr (!SK) {
      return false;
    } else {
      if (!sk_pending) return false;
      sk_pending = false;
      const int R = p.sk_tiles, G = p.sk_grid, b = blockIdx.x;
      const int j = static_cast<int>(static_cast<long long>(b) * R / G);
      const int f = sk_first_cta(j, R, G), n = sk_first_cta(j + 1, R, G) - f;
      int kb0, kb1;
      sk_share(b - f, n, p.nkb, kb0, kb1);
      if (kb0 == kb1) return false;                 // more CTAs than slices in this group
      w = {p.dp_tiles + j, kb0, kb1, n == 1 ? -1 : 0};
      return true;
    }
  }
};

// Shared memory of one CTA.  The expert tables exist only in the grouped
// kernels and the column-scale ring only in tile mode (BTILE), so that each
// variant stays within the 227 KB a CTA may use.
template <bool GROUPED, bool BTILE>
struct SmemT {
  uint8_t a[STAGES][A_BYTES];     // 1024-byte aligned (offset 0)
  uint8_t b[STAGES][B_BYTES];
  // output staging of the promotion warps: warp w stages in bytes [2 KB w, 2 KB (w+1))
  alignas(1024) uint8_t cst[NUM_EPI_WARPS][CST_BYTES];
  // tile mode: the B column scales of SB slices of the current tile, [slice][column],
  // and the A row scales of the same slices, [slice][row]
  float sring[BTILE ? SB_SLOTS : 1][BTILE ? SB : 1][BTILE ? BN : 1];
  float saring[BTILE ? SB_SLOTS : 1][BTILE ? SB : 1][BTILE ? BM : 1];
  uint64_t full_bar[STAGES];
  uint64_t empty_bar[STAGES];
  uint64_t tfull_bar[2];
  uint64_t tempty_bar[2];
  uint64_t sfull_bar[SB_SLOTS];   // tile mode: ring slot written by the scale warp
  uint64_t sempty_bar[SB_SLOTS];  // tile mode: ring slot read by all promotion warps
  uint64_t drain_bar;
  uint32_t tmem_base;
  int abort_flag;
  int bad_offsets;
  int num_tiles;
  float amx[2][4][32];            // SwiGLU: per-row tile amax of each half (warp pairs)
  int cum[GROUPED ? MAX_EXPERTS + 1 : 1];    // grouped: tile prefix per expert
  int row0[GROUPED ? MAX_EXPERTS + 1 : 1];   // grouped: copy of offsets
};

using SmemDense = SmemT<false, false>;
using SmemGrouped = SmemT<true, false>;
using SmemTile = SmemT<false, true>;
static_assert(offsetof(SmemDense, cst) % 1024 == 0, "swizzled TMA staging is 1024-byte aligned");
static_assert(offsetof(SmemGrouped, cst) % 1024 == 0, "swizzled TMA staging is 1024-byte aligned");
static_assert(offsetof(SmemTile, cst) % 1024 == 0, "swizzled TMA staging is 1024-byte aligned");
static_assert(CST_BYTES == 32 * CST_ROW, "one staged chunk: 32 rows");
static_assert(offsetof(SmemTile, full_bar) % 8 == 0, "mbarriers are 8-byte aligned");
static_assert(offsetof(SmemGrouped, full_bar) % 8 == 0, "mbarriers are 8-byte aligned");
static_assert(offsetof(SmemTile, sring) % 16 == 0, "scale ring read as 16-byte pairs");
template <bool GROUPED, bool BTILE>
constexpr size_t smem_bytes() { return sizeof(SmemT<GROUPED, BTILE>) + 1024; }
static_assert(smem_bytes<false, true>() <= 232448 && smem_bytes<true, false>() <= 232448 &&
                  smem_bytes<false, false>() <= 232448,
              "a CTA may use at most 227 KB of shared memory");

struct Tile {
  int m0;       // first row of A / C
  int row_end;  // rows >= row_end are not stored (expert end or M)
  int n0;       // first column
  int e;        // expert (0 when dense)
};

// Tile t of a dense launch: groups of group_m M-tiles, all N-tiles of a group
// before the next group, M fastest inside a group.
__host__ __device__ __forceinline__ Tile dense_tile(int t, const GemmParams& p) {
  Tile r;
  const int group = p.group_m * p.n_tiles;
  const int g = t / group;
  const int first = g * p.group_m;
  const int gm = min(p.group_m, p.m_tiles - first);
  const int local = t - g * group;
  const int mb = first + local % gm;
  const int nb = local / gm;
  r.m0 = mb * BM;
  r.row_end = p.M;
  r.n0 = nb * BN;
  r.e = 0;
  return r;
}

template <bool GROUPED, class S>
__device__ __forceinline__ Tile tile_of(int t, const GemmParams& p, const S& sm) {
  Tile r;
  if constexpr (!GROUPED) {
    r = dense_tile(t, p);
  } else {
    // largest e with cum[e] <= t (experts with no tiles have cum[e] == cum[e+1])
    int lo = 0, hi = p.E - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (sm.cum[mid] <= t) lo = mid; else hi = mid - 1;
    }
    const int e = lo;
    const int rows = sm.row0[e + 1] - sm.row0[e];
    const int mt = (rows + BM - 1) / BM;
    const int local = t - sm.cum[e];
    const int nb = local / mt;
    const int mb = local - nb * mt;
    r.m0 = sm.row0[e] + mb * BM;
    r.row_end = sm.row0[e + 1];
    r.n0 = nb * BN;
    r.e = e;
  }
  return r;
}

// Limit of the waits that let a stopping CTA's own TMA copies and MMAs finish
// before it releases its shared memory and TMEM: at least 2^27 cycles
// (~67 ms), whatever limit the caller set for the pipeline waits, so that a
// small limit cannot make a CTA leave with work still landing.
__device__ __forceinline__ long long teardown_limit(long long wait_limit) {
  constexpr long long kMin = 1ll << 27;
  return wait_limit > kMin ? wait_limit : kMin;
}

template <bool GROUPED, bool BTILE, int EPI, bool SK = false>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    blockscaled_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                            const __grid_constant__ CUtensorMap tmB,
                            const __grid_constant__ CUtensorMap tmC,
                            const __grid_constant__ CUtensorMap tmW, const GemmParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte alignment of the operand stages (required by the 128B swizzle)
  using Smem = SmemT<GROUPED, BTILE>;
  // SK: the split launch of a stream-K GEMM (dense kernels that store C
  // only).  It runs after the launch of the whole tiles, which lets it start
  // as soon as each of its CTAs leaves (programmatic dependent launch); that
  // launch's loops keep the slice bounds 0..nkb of a kernel without the split.
  constexpr bool SKOK = SK && !GROUPED && EPI == EPI_STORE;
  if constexpr (!GROUPED && EPI == EPI_STORE && !SK) griddep_launch_dependents();
  Smem& sm = *reinterpret_cast<Smem*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile int* abort_flag = &sm.abort_flag;

  // ---------------------------------------------------------------- set-up
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&sm.full_bar[s]), 1);
      mbar_init(smem_u32(&sm.empty_bar[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&sm.tfull_bar[b]), 1);
      mbar_init(smem_u32(&sm.tempty_bar[b]), NUM_EPI_WARPS);
    }
    for (int b = 0; b < SB_SLOTS; ++b) {
      mbar_init(smem_u32(&sm.sfull_bar[b]), 1);
      mbar_init(smem_u32(&sm.sempty_bar[b]), NUM_EPI_WARPS);
    }
    mbar_init(smem_u32(&sm.drain_bar), 1);
    fence_mbar_init();
    sm.abort_flag = 0;
    sm.bad_offsets = 0;
  }
  if (warp == PRODUCER_WARP && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmC);
    if (p.sk_tiles > 0) tma_prefetch_desc(&tmW);
  }
  if constexpr (GROUPED) {
    // Copy and check the offsets, then prefix the per-expert tile counts with
    // one warp: lane l owns a contiguous chunk of experts.
    if (warp == 0) {
      const int E = p.E;
      const int per = (E + 31) / 32;
      const int e0 = min(E, lane * per), e1 = min(E, e0 + per);
      int bad = 0, local = 0;
      for (int e = e0; e < e1; ++e) {
        const int r0 = p.offsets[e], r1 = p.offsets[e + 1];
        sm.row0[e] = r0;
        if (r1 < r0 || r0 < 0 || r1 > p.M) bad = 1;
        local += ((r1 - r0) + BM - 1) / BM * p.n_tiles;
      }
      int incl = local;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int v = __shfl_up_sync(0xFFFFFFFFu, incl, off);
        if (lane >= off) incl += v;
      }
      int run = incl - local;
      for (int e = e0; e < e1; ++e) {
        sm.cum[e] = run;
        const int r0 = p.offsets[e], r1 = p.offsets[e + 1];
        run += max(0, (r1 - r0) + BM - 1) / BM * p.n_tiles;
      }
      bad = __any_sync(0xFFFFFFFFu, bad);
      if (lane == 31) sm.num_tiles = incl;
      if (lane == 0) {
        sm.row0[E] = p.offsets[E];
        if (p.offsets[0] != 0 || p.offsets[E] != p.M) bad = 1;
        sm.cum[E] = 0;
        sm.bad_offsets = bad;
      }
    }
  } else {
    if (threadIdx.x == 0) sm.num_tiles = p.m_tiles * p.n_tiles;
  }
  if (warp == MMA_WARP) {
    tmem_alloc(smem_u32(&sm.tmem_base), TMEM_COLS);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = sm.tmem_base;
  const bool bad = GROUPED && sm.bad_offsets;
  if (bad && threadIdx.x == 0) record_status(p.status, FP8FG_ERR_BAD_OFFSETS);
  const int num_tiles = bad ? 0 : sm.num_tiles;
  const int nkb = p.nkb;

  if (warp >= NUM_EPI_WARPS) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(regs_producer(GROUPED, EPI)));
    if (warp == PRODUCER_WARP) {
      // ------------------------------------------------------- TMA producer
      if (lane == 0) {
        int stage = 0;
        uint32_t phase = 0;
        uint32_t issued = 0, issued_parity = 0;   // per-stage bits
        WorkList<SKOK> wl;
        wl.init(p);
        Work wk;
        while (!*abort_flag && wl.next(p, num_tiles, wk)) {
          const Tile tl = tile_of<GROUPED>(wk.t, p, sm);
          for (int kb = wk.kb0; kb < wk.kb1; ++kb) {
            if (!mbar_wait(smem_u32(&sm.empty_bar[stage]), phase ^ 1, p.wait_limit, abort_flag,
                           p.status))
              break;
            const uint32_t fb = smem_u32(&sm.full_bar[stage]);
            mbar_arrive_expect_tx(fb, A_BYTES + B_BYTES);
            tma_load_2d(smem_u32(sm.a[stage]), &tmA, fb, kb * BK, tl.m0);
            if constexpr (EPI == EPI_SWIGLU) {
              // B rows of the stage: gate j0..j0+63, up j0.., gate j0+64.., up j0+64..
              // (j0 = n0/2), so each TMEM column half holds g and u of the same
              // 64 outputs.  One request over the 5-D view {K, 64 rows, gate/up,
              // 64-row block, expert} of B lands them in that order (four
              // 64-row requests measured 5 % slower for the kernel).
              tma_load_5d(smem_u32(sm.b[stage]), &tmB, fb, kb * BK, 0, 0, tl.n0 / 128, tl.e);
            } else if constexpr (GROUPED)
              tma_load_3d(smem_u32(sm.b[stage]), &tmB, fb, kb * BK, tl.n0, tl.e);
            else
              tma_load_2d(smem_u32(sm.b[stage]), &tmB, fb, kb * BK, tl.n0);
            issued |= 1u << stage;
            issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
            if (++stage == STAGES) { stage = 0; phase ^= 1; }
          }
        }
        // never leave the CTA with a bulk copy still landing in shared memory
        volatile int never = 0;
        for (int s = 0; s < STAGES; ++s)
          if (issued & (1u << s))
            mbar_wait(smem_u32(&sm.full_bar[s]), (issued_parity >> s) & 1, teardown_limit(p.wait_limit), &never,
                      p.status);
      }
    } else if (warp == MMA_WARP) {
      // --------------------------------------------------------- MMA issuer
      // The whole warp runs the loop: lane 0 waits on the barriers and
      // broadcasts the outcome, one elected lane issues.
      int stage = 0;
      uint32_t phase = 0;
      uint32_t it = 0;                              // slice counter (TMEM buffers)
      uint32_t tcount = 0;                          // tile counter (study mode buffers)
      bool ok = true;
      WorkList<SKOK> wl;
      wl.init(p);
      Work wk;
      while (ok && wl.next(p, num_tiles, wk)) {
        for (int kb = wk.kb0; kb < wk.kb1; ++kb, ++it) {
          const uint32_t ix = EPI == EPI_WHOLEK ? tcount : it;
          const uint32_t buf = ix & 1, bpar = (ix >> 1) & 1;
          int got = 0;
          if (lane == 0)
            got = (EPI != EPI_WHOLEK || kb == 0
                       ? mbar_wait(smem_u32(&sm.tempty_bar[buf]), bpar ^ 1, p.wait_limit,
                                   abort_flag, p.status)
                       : true) &&
                  mbar_wait(smem_u32(&sm.full_bar[stage]), phase, p.wait_limit, abort_flag,
                            p.status);
          if (!__shfl_sync(0xFFFFFFFFu, got, 0)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sm.a[stage]);
          const uint32_t b0 = smem_u32(sm.b[stage]);
          const uint32_t d = tmem_base + buf * BN;
#pragma unroll
          for (int k = 0; k < BK / 32; ++k)
            mma_f8_elect(d, smem_desc_sw128(a0 + 32 * k), smem_desc_sw128(b0 + 32 * k), IDESC,
                         k > 0 || (EPI == EPI_WHOLEK && kb > 0) ? 1u : 0u);
          mma_commit_elect(smem_u32(&sm.empty_bar[stage]));
          if (EPI != EPI_WHOLEK || kb == nkb - 1) mma_commit_elect(smem_u32(&sm.tfull_bar[buf]));
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
        ++tcount;
      }
      // all issued MMAs must finish before TMEM is released
      mma_commit_elect(smem_u32(&sm.drain_bar));
      if (lane == 0) {
        volatile int never = 0;
        mbar_wait(smem_u32(&sm.drain_bar), 0, teardown_limit(p.wait_limit), &never, p.status);
      }
    } else if (BTILE && warp == SCALE_WARP) {
      // ----------------------------------------------- tile-mode scale loader
      // For every SB slices of a tile, the 256 column scales sb[n0 + c, kb]
      // (c = lane + 32 i) are read and written transposed, [slice][column],
      // into a ring slot that the promotion warps read as 16-byte column
      // pairs, and the 128 row scales sa[m0 + r, kb] likewise, [slice][row].
      // Columns past N and rows past M read the last column's and row's
      // scales (never stored).
      uint32_t grp = 0;
      bool live = true;
      WorkList<SKOK> wl;
      wl.init(p);
      Work wk;
      while (live && wl.next(p, num_tiles, wk)) {
        const Tile tl = tile_of<GROUPED>(wk.t, p, sm);
        for (int kb0 = wk.kb0; kb0 < wk.kb1; kb0 += SB, ++grp) {
          const uint32_t slot = grp % SB_SLOTS;
          if (!mbar_wait(smem_u32(&sm.sempty_bar[slot]), ((grp / SB_SLOTS) & 1) ^ 1, p.wait_limit,
                         abort_flag, p.status)) {
            live = false;
            break;
          }
#pragma unroll
          for (int i = 0; i < BN / 32; ++i) {
            const int c = lane + 32 * i;
            const float* col = p.sb + static_cast<int64_t>(min(tl.n0 + c, p.N - 1)) * nkb;
#pragma unroll
            for (int q = 0; q < SB; ++q)
              sm.sring[slot][q][c] = kb0 + q < wk.kb1 ? __ldg(col + kb0 + q) : 0.0f;
          }
#pragma unroll
          for (int i = 0; i < BM / 32; ++i) {
            const int r = lane + 32 * i;
            const float* rw = p.sa + static_cast<int64_t>(min(tl.m0 + r, p.M - 1)) * nkb;
#pragma unroll
            for (int q = 0; q < SB; ++q)
              sm.saring[slot][q][r] = kb0 + q < wk.kb1 ? __ldg(rw + kb0 + q) : 0.0f;
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&sm.sfull_bar[slot]));
        }
      }
    }
  } else {
    // ------------------------------------------------ promotion + epilogue
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(regs_epilogue(GROUPED, EPI)));
    const int quad = warp & 3;                      // TMEM lane quadrant
    const int half = warp >> 2;                     // N half of the tile
    const int n_blocks = p.N / 128;                 // block-mode scale rows per expert
    const uint32_t lane_taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + half * 128;
    uint32_t it = 0;
    uint32_t tcount = 0;                            // tile counter (study mode buffers)
    uint32_t sgrp = 0;                              // tile mode: scale-ring group counter
    bool staged = false;                            // a store of this warp may still read cst
    bool ok = true;
    WorkList<SKOK> wl;
    wl.init(p);
    Work wk;
    while (ok && wl.next(p, num_tiles, wk)) {
      const Tile tl = tile_of<GROUPED>(wk.t, p, sm);
      const int row = tl.m0 + quad * 32 + lane;
      const bool row_ok = row < tl.row_end;
      const int col_h = tl.n0 + half * 128;         // first column of this half
      const bool half_ok = col_h < p.N;
      // rows and columns past the end read valid scales (row 0 / the last
      // column) and are never stored
      const float* sa_row = p.sa + static_cast<int64_t>(row_ok ? row : 0) * nkb;
      // B row of this half's first column (SwiGLU: the gate block j0 = n0/2;
      // the up block is I/128 blocks further, see the K loop)
      const int brow_h = EPI == EPI_SWIGLU ? tl.n0 / 2 : col_h;
      const float* sb_ptr =
          p.sb + (static_cast<int64_t>(tl.e) * n_blocks + (half_ok ? brow_h / 128 : 0)) * nkb;

      uint64_t acc[64];
#pragma unroll
      for (int j = 0; j < 64; ++j) acc[j] = 0;

      if constexpr (BTILE) {
        // Row and column scales come from the scale warp's ring: each slot
        // holds SB slices of this tile's 128 row and 256 column scales; a warp
        // waits for a slot before its first slice and frees it after its
        // last, so no barrier joins the promotion warps and they issue no
        // global loads.
        for (int kb = wk.kb0; kb < wk.kb1; ++kb, ++it) {
          const uint32_t slot = sgrp % SB_SLOTS;
          const int g = kb - wk.kb0;                  // slice within the unit (ring groups start at kb0)
          if (g % SB == 0 && !mbar_wait(smem_u32(&sm.sfull_bar[slot]), (sgrp / SB_SLOTS) & 1,
                                        p.wait_limit, abort_flag, p.status)) {
            ok = false;
            break;
          }
          const float sa_cur = sm.saring[slot][g % SB][quad * 32 + lane];
          const uint32_t buf = it & 1, bpar = (it >> 1) & 1;
          if (!mbar_wait(smem_u32(&sm.tfull_bar[buf]), bpar, p.wait_limit, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t taddr = lane_taddr + buf * BN;
          const uint64_t sa2 = pack2(__float_as_uint(sa_cur), __float_as_uint(sa_cur));
          const uint32_t sbv = smem_u32(&sm.sring[slot][g % SB][half * 128]);
          // Eight chunks of 16 columns, software-pipelined: chunk c + 1's TMEM
          // load and column scales (read as pairs) are in flight while chunk
          // c's coefficients sa * sb[col] and FMAs issue.
          uint32_t r[2][16];
          uint64_t q[8];
          tmem_ld_16cols(taddr, r[0]);
#pragma unroll
          for (int j = 0; j < 4; ++j) lds_2x64(sbv + 16 * j, q[2 * j], q[2 * j + 1]);
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            uint64_t cf[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) cf[j] = mul2_s(q[j], sa2);
            if (c + 1 < 8) {
#pragma unroll
              for (int j = 0; j < 4; ++j)
                lds_2x64(sbv + ((c + 1) * 16 + 4 * j) * 4, q[2 * j], q[2 * j + 1]);
            }
            tmem_ld_wait_regs(r[c & 1]);
            if (c + 1 < 8) tmem_ld_16cols(taddr + (c + 1) * 16, r[(c + 1) & 1]);
#pragma unroll
            for (int j = 0; j < 8; ++j)
              fma2_s(acc[c * 8 + j], pack2(r[c & 1][2 * j], r[c & 1][2 * j + 1]), cf[j]);
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&sm.tempty_bar[buf]));
          if (g % SB == SB - 1 || kb == wk.kb1 - 1) {
            // this warp's reads of the slot are complete (their values were used above)
            if (lane == 0) mbar_arrive(smem_u32(&sm.sempty_bar[slot]));
            ++sgrp;
          }
        }
        if (!ok) break;
      } else if constexpr (EPI == EPI_WHOLEK) {
        // the whole K sum of this tile sits in buffer tcount % 2: scale it once
        const float s = __ldg(p.sa) * __ldg(p.sb);
        const uint64_t s2 = pack2(__float_as_uint(s), __float_as_uint(s));
        const uint32_t buf = tcount & 1, bpar = (tcount >> 1) & 1;
        ++tcount;
        if (!mbar_wait(smem_u32(&sm.tfull_bar[buf]), bpar, p.wait_limit, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t taddr = lane_taddr + buf * BN;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t r[32];
          tmem_ld_32cols(taddr + c * 32, r);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) fma2(acc[c * 16 + j], pack2(r[2 * j], r[2 * j + 1]), s2);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sm.tempty_bar[buf]));
      } else {
        // SwiGLU: columns 64..127 of the half are up rows, whose block scale
        // lies I/128 blocks after the gate block
        const float* sbu_ptr = sb_ptr + (EPI == EPI_SWIGLU ? (p.N / 256) * nkb : 0);
        float sa_next = __ldg(sa_row + wk.kb0);
        float sb_next = __ldg(sb_ptr + wk.kb0);
        float sbu_next = EPI == EPI_SWIGLU ? __ldg(sbu_ptr + wk.kb0) : 0.0f;
        for (int kb = wk.kb0; kb < wk.kb1; ++kb, ++it) {
          const float sa_cur = sa_next, sb_cur = sb_next, sbu_cur = sbu_next;
          if (kb + 1 < wk.kb1) {
            sa_next = __ldg(sa_row + kb + 1);
            sb_next = __ldg(sb_ptr + kb + 1);
            if constexpr (EPI == EPI_SWIGLU) sbu_next = __ldg(sbu_ptr + kb + 1);
          }
          const uint32_t buf = it & 1, bpar = (it >> 1) & 1;
          if (!mbar_wait(smem_u32(&sm.tfull_bar[buf]), bpar, p.wait_limit, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t taddr = lane_taddr + buf * BN;
          const float s = sa_cur * sb_cur;
          const uint64_t s2 = pack2(__float_as_uint(s), __float_as_uint(s));
          const float su = sa_cur * sbu_cur;
          const uint64_t su2 = pack2(__float_as_uint(su), __float_as_uint(su));
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t r[32];
            tmem_ld_32cols(taddr + c * 32, r);
            tmem_ld_wait();
            const uint64_t sc2 = EPI == EPI_SWIGLU && c >= 2 ? su2 : s2;
#pragma unroll
            for (int j = 0; j < 16; ++j) fma2(acc[c * 16 + j], pack2(r[2 * j], r[2 * j + 1]), sc2);
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&sm.tempty_bar[buf]));
        }
        if constexpr (EPI == EPI_SWIGLU) {
          // the gate/up warp pair meets at the exchange below: both leave
          // together if either one's K loop gave up
          if (bar_any(3 + quad, 64, !ok)) {
            ok = false;
            break;
          }
        } else if (!ok) {
          break;
        }
      }

      if constexpr (EPI == EPI_SWIGLU) {
        // --- grouped SwiGLU: this thread holds g (accumulator pairs 0..31) and
        // u (pairs 32..63) of outputs j0 + 64*half .. +63 of its row.  It forms
        // h = silu(g) * u in FP32 (the exact-silu version measured ~10 % slower
        // for the whole kernel), the warp pair (same rows, both halves)
        // combines the 1x128 tile amax through shared memory, and each thread
        // stores its 64 codes; half 0 stores the tile's scale.  Rows past the
        // expert's end are not stored.
        float amax = 0.0f;
#pragma unroll
        for (int v = 0; v < 32; ++v) {
          float g0, g1, u0, u1;
          unpack2(acc[v], g0, g1);
          unpack2(acc[32 + v], u0, u1);
          // silu with the fast exponential and divide: relative error at most
          // (4 + 1.2 |g|) 2^-23 by their documented bounds (2 + 1.173 |x| ulp and
          // 2 ulp); below g = -87 the divide returns a zero of the right sign
          const float h0 = __fmul_rn(__fdividef(g0, __fadd_rn(1.0f, __expf(-g0))), u0);
          const float h1 = __fmul_rn(__fdividef(g1, __fadd_rn(1.0f, __expf(-g1))), u1);
          acc[v] = pack2(__float_as_uint(h0), __float_as_uint(h1));
          amax = fmaxf(amax, fmaxf(fabsf(h0), fabsf(h1)));
        }
        // amax slots: [half][quad][lane]; the partner's slot is rewritten only
        // after the next tile's pair vote, which follows this read
        sm.amx[half][quad][lane] = amax;
        bar_sync(3 + quad, 64);
        amax = fmaxf(amax, sm.amx[half ^ 1][quad][lane]);
        const Scale sc = scale_from_amax(amax, p.pow2_out != 0);
        const int I = p.N / 2;
        const int j0 = tl.n0 / 2;
        if (half == 0 && row_ok) p.s_out[static_cast<int64_t>(row) * (I / 128) + j0 / 128] = sc.s;
        // the row's 64 codes are one 64-byte staging row: a warp whose rows lie
        // inside the expert (or end at M) writes them with one TMA tile store
        const int wrow0 = tl.m0 + quad * 32;
        const bool whole = wrow0 + 32 <= tl.row_end || tl.row_end == p.M;
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 4; ++i)               // 16 codes = outputs 16i .. 16i+15
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            float x0, x1, x2, x3;
            unpack2(acc[8 * i + 2 * k], x0, x1);
            unpack2(acc[8 * i + 2 * k + 1], x2, x3);
            w[4 * i + k] = e4m3x2(__fmul_rn(x0, sc.m), __fmul_rn(x1, sc.m)) |
                           (e4m3x2(__fmul_rn(x2, sc.m), __fmul_rn(x3, sc.m)) << 16);
          }
        if (whole && wrow0 < tl.row_end) {
          uint32_t wl = (warp << 8) | lane;
          asm volatile("" : "+r"(wl));
          const uint32_t cbuf = smem_u32(sm.cst[0]) + (wl >> 8) * CST_BYTES;
          const uint32_t srow = cbuf + (wl & 31) * CST_ROW;
          const uint32_t swz = ((wl & 31) >> 1) & 3;
          if (staged) {
            if (lane == 0) bulk_wait_read_all();
            __syncwarp();
          }
#pragma unroll
          for (int u = 0; u < 4; ++u)
            sts_128(srow + ((u ^ swz) << 4), w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&tmC, cbuf, j0 + 64 * half, wrow0);
            bulk_commit();
          }
          staged = true;
        } else if (row_ok) {
          uint8_t* dst = static_cast<uint8_t*>(p.c) + static_cast<int64_t>(row) * I + j0 + 64 * half;
#pragma unroll
          for (int i = 0; i < 4; ++i)
            *reinterpret_cast<uint4*>(dst + 16 * i) =
                make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
        }
      } else if constexpr (GROUPED) {
        // --- grouped: a warp whose 32 rows lie inside the expert (or end at M,
        // where the store clips) writes through the swizzled staging and TMA
        // tile stores like the dense kernel; a warp whose rows run past the
        // expert's end (the rows after belong to the next expert) stores its
        // valid rows per thread.
        const int wrow0 = tl.m0 + quad * 32;
        const bool whole = wrow0 + 32 <= tl.row_end || tl.row_end == p.M;
        if (half_ok && wrow0 < tl.row_end && whole) {
          uint32_t wl = (warp << 8) | lane;
          asm volatile("" : "+r"(wl));
          const uint32_t cbuf = smem_u32(sm.cst[0]) + (wl >> 8) * CST_BYTES;
          const uint32_t srow = cbuf + (wl & 31) * CST_ROW;
          const uint32_t swz = ((wl & 31) >> 1) & 3;
          const int W = p.c_f32 ? 16 : 32;        // columns per chunk
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            if (p.c_f32 || q < 4) {
              if (staged) {
                if (lane == 0) bulk_wait_read_all();
                __syncwarp();
              }
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                uint32_t w[4];
                if (p.c_f32) {
                  const uint64_t x0 = acc[8 * q + 2 * u], x1 = acc[8 * q + 2 * u + 1];
                  w[0] = static_cast<uint32_t>(x0);
                  w[1] = static_cast<uint32_t>(x0 >> 32);
                  w[2] = static_cast<uint32_t>(x1);
                  w[3] = static_cast<uint32_t>(x1 >> 32);
                } else {
#pragma unroll
                  for (int i = 0; i < 4; ++i) {
                    float lo, hi;
                    unpack2(acc[(16 * q + 4 * u + i) & 63], lo, hi);
                    const __nv_bfloat162 b2 = __floats2bfloat162_rn(lo, hi);
                    w[i] = *reinterpret_cast<const uint32_t*>(&b2);
                  }
                }
                sts_128(srow + ((u ^ swz) << 4), w[0], w[1], w[2], w[3]);
              }
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                tma_store_2d(&tmC, cbuf, col_h + q * W, wrow0);
                bulk_commit();
              }
              staged = true;
            }
          }
        } else if (row_ok && half_ok) {
          if (p.c_f32) {
            float* dst = static_cast<float*>(p.c) + static_cast<int64_t>(row) * p.N + col_h;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              float x0, x1, x2, x3;
              unpack2(acc[2 * j], x0, x1);
              unpack2(acc[2 * j + 1], x2, x3);
              *reinterpret_cast<float4*>(dst + 4 * j) = make_float4(x0, x1, x2, x3);
            }
          } else {
            __nv_bfloat16* dst =
                static_cast<__nv_bfloat16*>(p.c) + static_cast<int64_t>(row) * p.N + col_h;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              uint32_t w[4];
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                float lo, hi;
                unpack2(acc[4 * j + i], lo, hi);
                const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
                w[i] = *reinterpret_cast<const uint32_t*>(&v);
              }
              *reinterpret_cast<uint4*>(dst + 8 * j) = make_uint4(w[0], w[1], w[2], w[3]);
            }
          }
        }
      } else if constexpr (EPI == EPI_QUANT) {
        // --- dense, E4M3 output: the thread's 128 columns of its row are one
        // 1x128 tile; the same amax/scale/multiplier rules as act_quant apply
        // to the FP32 accumulator, and the codes leave like the BF16 output
        // (two 64-byte chunks per row through the swizzled staging).
        const int wrow0 = tl.m0 + quad * 32;
        if (half_ok && wrow0 < p.M) {
          float amax = 0.0f;
#pragma unroll
          for (int j = 0; j < 64; ++j) {
            float lo, hi;
            unpack2(acc[j], lo, hi);
            amax = fmaxf(amax, fmaxf(fabsf(lo), fabsf(hi)));
          }
          const Scale sc = scale_from_amax(amax, p.pow2_out != 0);
          if (row < p.M) p.s_out[static_cast<int64_t>(row) * (p.N / 128) + col_h / 128] = sc.s;
          uint32_t wl = (warp << 8) | lane;
          asm volatile("" : "+r"(wl));
          const uint32_t cbuf = smem_u32(sm.cst[0]) + (wl >> 8) * CST_BYTES;
          const uint32_t srow = cbuf + (wl & 31) * CST_ROW;
          const uint32_t swz = ((wl & 31) >> 1) & 3;
#pragma unroll
          for (int q = 0; q < 2; ++q) {           // 64 codes per chunk
            if (staged) {
              if (lane == 0) bulk_wait_read_all();
              __syncwarp();
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              uint32_t w[4];
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                // columns 64q + 16u + 4i .. +3 = accumulator pairs 32q + 8u + 2i, +1
                float x0, x1, x2, x3;
                unpack2(acc[32 * q + 8 * u + 2 * i], x0, x1);
                unpack2(acc[32 * q + 8 * u + 2 * i + 1], x2, x3);
                w[i] = e4m3x2(__fmul_rn(x0, sc.m), __fmul_rn(x1, sc.m)) |
                       (e4m3x2(__fmul_rn(x2, sc.m), __fmul_rn(x3, sc.m)) << 16);
              }
              sts_128(srow + ((u ^ swz) << 4), w[0], w[1], w[2], w[3]);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmC, cbuf, col_h + 64 * q, wrow0);
              bulk_commit();
            }
            staged = true;
          }
        }
      } else {
        // --- dense: the warp's 32 rows x 128 columns of its half go out in
        // chunks of 64 bytes per row.  Chunk q of row `lane` goes to staging
        // row `lane`, its 16-byte unit u at unit u ^ ((lane/2) % 4) (the 64-byte
        // swizzle), so a warp's st.shared.v4 hits every bank once per 8 lanes;
        // one TMA store writes the chunk and clips rows at or past M.  A part
        // of a tile shared between CTAs (stream-K) goes whole, in FP32, to this
        // CTA's workspace slot instead, for the fix-up kernel to add up.
        const bool partial = wk.slot >= 0;
        const bool f32 = partial || p.c_f32;
        const int wrow0 = partial ? static_cast<int>(blockIdx.x) * BM + quad * 32 : tl.m0 + quad * 32;
        const int wcol0 = partial ? half * 128 : col_h;
        if (partial || (half_ok && wrow0 < p.M)) {
          // formed here rather than hoisted out of the tile loop, so that they
          // hold no registers during the K loop
          uint32_t wl_ = (warp << 8) | lane;
          asm volatile("" : "+r"(wl_));
          const uint32_t cbuf = smem_u32(sm.cst[0]) + (wl_ >> 8) * CST_BYTES;
          const uint32_t srow = cbuf + (wl_ & 31) * CST_ROW;
          const uint32_t swz = ((wl_ & 31) >> 1) & 3;
          const int W = f32 ? 16 : 32;             // columns per chunk
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            if ((f32 || q < 4) && (partial || col_h + q * W < p.N)) {
              if (staged) {
                if (lane == 0) bulk_wait_read_all();
                __syncwarp();
              }
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                uint32_t w[4];
                if (f32) {
                  // columns 16q + 4u .. +3 = accumulator pairs 8q + 2u, +1
                  const uint64_t x0 = acc[8 * q + 2 * u], x1 = acc[8 * q + 2 * u + 1];
                  w[0] = static_cast<uint32_t>(x0);
                  w[1] = static_cast<uint32_t>(x0 >> 32);
                  w[2] = static_cast<uint32_t>(x1);
                  w[3] = static_cast<uint32_t>(x1 >> 32);
                } else {
                  // columns 32q + 8u .. +7 = accumulator pairs 16q + 4u .. +3
#pragma unroll
                  for (int i = 0; i < 4; ++i) {
                    float lo, hi;
                    unpack2(acc[(16 * q + 4 * u + i) & 63], lo, hi);
                    const __nv_bfloat162 b2 = __floats2bfloat162_rn(lo, hi);
                    w[i] = *reinterpret_cast<const uint32_t*>(&b2);
                  }
                }
                sts_128(srow + ((u ^ swz) << 4), w[0], w[1], w[2], w[3]);
              }
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                tma_store_2d(partial ? &tmW : &tmC, cbuf, wcol0 + q * W, wrow0);
                bulk_commit();
              }
              staged = true;
            }
          }
        }
      }
    }
    // the CTA's shared memory must outlive the reads of the last stores
    if (lane == 0) bulk_wait_all();
  }

  // -------------------------------------------------------------- teardown
  __syncthreads();
  if (warp == MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
  // the split launch ends only after the whole-tile launch it overlaps, so
  // that work queued after the GEMM sees all of C
  if constexpr (SKOK) griddep_wait();
}

// Stream-K fix-up: one thread per four columns of a row of a split tile,
// BM * BN / (4 * kFixupThreads) CTAs per tile.  The tile's group of CTAs is
// recomputed from the same split as in WorkList; a tile with a single member
// was stored by it and is skipped.  Members whose share is empty (only when a
// group has more CTAs than slices) wrote nothing and are skipped.  The
// members' partial sums are added in CTA order (FP32, so the result does not
// depend on timing), loaded eight at a time so that the loads overlap, and
// the tile is written to C, clipped at M and N.
constexpr int kFixupThreads = 256;
constexpr int kFixupCtasPerTile = BM * BN / 4 / kFixupThreads;
static_assert(kFixupCtasPerTile * kFixupThreads * 4 == BM * BN, "fix-up covers the tile");

template <bool F32OUT>
__global__ void __launch_bounds__(kFixupThreads) streamk_fixup_kernel(const float* __restrict__ ws,
                                                                      void* __restrict__ c,
                                                                      const GemmParams p) {
  const int j = blockIdx.x;
  const int R = p.sk_tiles, G = p.sk_grid;
  const int f = sk_first_cta(j, R, G), n = sk_first_cta(j + 1, R, G) - f;
  if (n == 1) return;
  const Tile tl = dense_tile(p.dp_tiles + j, p);
  const int idx = blockIdx.y * kFixupThreads + threadIdx.x;   // float4 of the tile
  const int r = idx / (BN / 4), cg = (idx % (BN / 4)) * 4;
  const int row = tl.m0 + r, col = tl.n0 + cg;
  if (row >= p.M || col >= p.N) return;       // N % 16 == 0: four columns are in or out together
  const float4* src =
      reinterpret_cast<const float4*>(ws + (static_cast<long long>(f) * BM + r) * BN + cg);
  constexpr long long kSlot4 = static_cast<long long>(BM) * BN / 4;   // one member's slot
  const bool may_be_empty = n > p.nkb;        // else every share holds a slice
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int i0 = 0; i0 < n; i0 += 8) {
    float4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u)
      v[u] = i0 + u < n ? __ldg(src + (i0 + u) * kSlot4) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (i0 + u >= n) break;
      if (may_be_empty) {
        int kb0, kb1;
        sk_share(i0 + u, n, p.nkb, kb0, kb1);
        if (kb0 == kb1) continue;
      }
      acc.x = __fadd_rn(acc.x, v[u].x);
      acc.y = __fadd_rn(acc.y, v[u].y);
      acc.z = __fadd_rn(acc.z, v[u].z);
      acc.w = __fadd_rn(acc.w, v[u].w);
    }
  }
  if constexpr (F32OUT) {
    *reinterpret_cast<float4*>(static_cast<float*>(c) + static_cast<long long>(row) * p.N + col) = acc;
  } else {
    const __nv_bfloat162 lo2 = __floats2bfloat162_rn(acc.x, acc.y);
    const __nv_bfloat162 hi2 = __floats2bfloat162_rn(acc.z, acc.w);
    uint2 v;
    v.x = *reinterpret_cast<const uint32_t*>(&lo2);
    v.y = *reinterpret_cast<const uint32_t*>(&hi2);
    *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(c) + static_cast<long long>(row) * p.N + col) = v;
  }
}

// One CTA waits on an mbarrier that nothing arrives on; the bounded wait must
// give up, record FP8FG_ERR_TIMEOUT and return.
__global__ void wait_timeout_selftest_kernel(long long limit, int* status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
    abort_flag = 0;
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(smem_u32(&bar), 0, limit, &abort_flag, status);
  __syncthreads();
}


bool make_maps(CUtensorMap* mA, CUtensorMap* mB, const uint8_t* a, int64_t rowsA,
               const uint8_t* b, int64_t E, int64_t N, int64_t K, uint32_t b_box_rows = BN) {
  const uint64_t dA[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(rowsA)};
  const uint64_t sA[1] = {static_cast<uint64_t>(K)};
  const uint32_t boxA[2] = {BK, BM};
  if (!encode_tensor_map_u8(mA, a, 2, dA, sA, boxA)) return false;
  if (E == 0) {
    const uint64_t dB[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(N)};
    const uint64_t sB[1] = {static_cast<uint64_t>(K)};
    const uint32_t boxB[2] = {BK, BN};
    return encode_tensor_map_u8(mB, b, 2, dB, sB, boxB);
  }
  const uint64_t dB[3] = {static_cast<uint64_t>(K), static_cast<uint64_t>(N),
                          static_cast<uint64_t>(E)};
  const uint64_t sB[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(N * K)};
  const uint32_t boxB[3] = {BK, b_box_rows, 1};
  return encode_tensor_map_u8(mB, b, 3, dB, sB, boxB);
}

// C [rows, N] row-major, stored by 32-row x 64-byte boxes (16 FP32 or 32 BF16
// columns) from 64-byte-swizzled staging.
bool make_c_map(CUtensorMap* mC, void* c, fp8fg_dtype ct, int64_t rows, int64_t N) {
  const bool f32 = ct == FP8FG_F32;
  const uint64_t elt = f32 ? 4 : 2;
  const uint64_t dC[2] = {static_cast<uint64_t>(N), static_cast<uint64_t>(rows)};
  const uint64_t sC[1] = {static_cast<uint64_t>(N) * elt};
  const uint32_t boxC[2] = {static_cast<uint32_t>(CST_ROW / elt), 32};
  return encode_tensor_map(mC, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                           c, 2, dC, sC, boxC, CU_TENSOR_MAP_SWIZZLE_64B);
}

// M-tiles per tile group of a dense launch: as many as keep the group's A rows
// within kGroupABytes, at least 8, at most all of them.
int group_m_tiles(int64_t m_tiles, int64_t K) {
  int64_t g = kGroupABytes / (static_cast<int64_t>(BM) * K);
  if (g < 8) g = 8;
  if (g > m_tiles) g = m_tiles;
  return static_cast<int>(g < 1 ? 1 : g);
}

template <bool GROUPED, bool BTILE, int EPI = EPI_STORE, bool SK = false>
cudaError_t set_smem_attr() {
  return set_max_dynamic_smem<blockscaled_gemm_kernel<GROUPED, BTILE, EPI, SK>>(
      static_cast<int>(smem_bytes<GROUPED, BTILE>()));
}

}  // namespace

namespace {

// Stream-K plan of a dense launch (see WorkList): tiles [0, dp_tiles) whole,
// the slices of the rest split evenly over `grid` CTAs.  Used when the last
// wave of whole tiles would leave at least kStreamKMinSlices slice-steps of
// most SMs idle (or when forced), and never in the whole-K study mode.
constexpr int kStreamKMinSlices = 40;

struct SplitPlan {
  int grid;
  int dp_tiles;
  int sk_tiles;
};

// The full waves stay whole tiles; each leftover tile is shared by a group of
// about sms / leftover CTAs (all tiles, when there are fewer tiles than SMs).
SplitPlan plan_split(int64_t tiles, int nkb, int sms, bool allow, bool force) {
  SplitPlan s{static_cast<int>(tiles < sms ? tiles : sms), INT32_MAX, 0};
  if (!allow || sms <= 0) return s;
  const int64_t rem = tiles % sms;
  if (rem == 0) return s;
  const int64_t idle_slices = (sms - rem) * static_cast<int64_t>(nkb) / sms;   // per SM, last wave
  if (!force && idle_slices < kStreamKMinSlices) return s;
  s.grid = sms;
  s.dp_tiles = static_cast<int>(tiles - rem);
  s.sk_tiles = static_cast<int>(rem);
  return s;
}

}  // namespace

size_t gemm_workspace_bytes(int64_t M, int64_t N, int64_t K, bool whole_k, bool force_sk) {
  const int64_t tiles = ((M + BM - 1) / BM) * ((N + BN - 1) / BN);
  const SplitPlan s = plan_split(tiles, static_cast<int>(K / BK), device_sm_count(), !whole_k, force_sk);
  if (s.sk_tiles == 0) return 0;
  return static_cast<size_t>(s.grid) * BM * BN * sizeof(float);
}

namespace {

// FP32 partial tiles of the stream-K workspace, [grid * BM rows, BN], stored
// like an FP32 C by 32-row x 64-byte boxes from 64-byte-swizzled staging.
bool make_ws_map(CUtensorMap* mW, float* ws, int grid) {
  const uint64_t dW[2] = {static_cast<uint64_t>(BN), static_cast<uint64_t>(grid) * BM};
  const uint64_t sW[1] = {static_cast<uint64_t>(BN) * 4};
  const uint32_t boxW[2] = {static_cast<uint32_t>(CST_ROW / 4), 32};
  return encode_tensor_map(mW, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, ws, 2, dW, sW, boxW,
                           CU_TENSOR_MAP_SWIZZLE_64B);
}

}  // namespace

fp8fg_status launch_gemm(const uint8_t* a, const float* sa, const uint8_t* b, const float* sb,
                         void* c, fp8fg_dtype ct, int64_t M, int64_t N, int64_t K, bool b_tile,
                         bool whole_k, void* ws, size_t ws_bytes, bool force_sk, cudaStream_t st) {
  CUtensorMap mA, mB, mC, mW;
  if (!make_maps(&mA, &mB, a, M, b, 0, N, K) || !make_c_map(&mC, c, ct, M, N))
    return FP8FG_ERR_CUDA;
  GemmParams p{};
  p.sa = sa;
  p.sb = sb;
  p.c = c;
  p.offsets = nullptr;
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.nkb = static_cast<int>(K / BK);
  p.m_tiles = static_cast<int>((M + BM - 1) / BM);
  p.n_tiles = static_cast<int>((N + BN - 1) / BN);
  p.group_m = group_m_tiles(p.m_tiles, K);
  p.E = 1;
  p.c_f32 = ct == FP8FG_F32;
  p.b_tile = b_tile ? 1 : 0;
  p.wait_limit = wait_limit_cycles();
  p.status = device_status_word();
  const int64_t tiles = static_cast<int64_t>(p.m_tiles) * p.n_tiles;
  // stream-K only with a workspace large enough for this device's split
  const size_t need = gemm_workspace_bytes(M, N, K, whole_k, force_sk);
  const bool sk = ws != nullptr && need > 0 && ws_bytes >= need;
  const SplitPlan plan = plan_split(tiles, p.nkb, device_sm_count(), sk, force_sk);
  p.dp_tiles = plan.dp_tiles;
  p.sk_tiles = plan.sk_tiles;
  p.sk_grid = plan.grid;
  if (plan.sk_tiles > 0) {
    if (!make_ws_map(&mW, static_cast<float*>(ws), plan.grid)) return FP8FG_ERR_CUDA;
  } else {
    mW = mC;                         // unused
  }
  const int grid = plan.grid;
  const bool split = plan.sk_tiles > 0;
  cudaError_t attr = whole_k  ? set_smem_attr<false, false, EPI_WHOLEK>()
                     : b_tile ? set_smem_attr<false, true>()
                              : set_smem_attr<false, false>();
  if (attr == cudaSuccess && split)
    attr = b_tile ? set_smem_attr<false, true, EPI_STORE, true>()
                  : set_smem_attr<false, false, EPI_STORE, true>();
  if (attr != cudaSuccess) return FP8FG_ERR_CUDA;
  if (whole_k) {
    blockscaled_gemm_kernel<false, false, EPI_WHOLEK>
        <<<grid, NUM_THREADS, smem_bytes<false, false>(), st>>>(mA, mB, mC, mW, p);
    return cudaGetLastError() == cudaSuccess ? FP8FG_OK : FP8FG_ERR_CUDA;
  }
  // whole tiles first; with a split, the tiles after them in a second launch
  // that may start on each SM as the first launch's CTA there leaves
  const bool whole = plan.dp_tiles > 0;
  if (whole) {
    if (b_tile)
      blockscaled_gemm_kernel<false, true, EPI_STORE>
          <<<grid, NUM_THREADS, smem_bytes<false, true>(), st>>>(mA, mB, mC, mW, p);
    else
      blockscaled_gemm_kernel<false, false, EPI_STORE>
          <<<grid, NUM_THREADS, smem_bytes<false, false>(), st>>>(mA, mB, mC, mW, p);
    if (cudaGetLastError() != cudaSuccess) return FP8FG_ERR_CUDA;
  }
  if (split) {
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(plan.grid));
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = b_tile ? smem_bytes<false, true>() : smem_bytes<false, false>();
    cfg.stream = st;
    // overlap only a launch of this GEMM: without one, the split launch
    // waits for all earlier work like any other launch
    cfg.attrs = whole ? pdl : nullptr;
    cfg.numAttrs = whole ? 1 : 0;
    const cudaError_t e =
        b_tile ? cudaLaunchKernelEx(&cfg, blockscaled_gemm_kernel<false, true, EPI_STORE, true>, mA,
                                    mB, mC, mW, p)
               : cudaLaunchKernelEx(&cfg, blockscaled_gemm_kernel<false, false, EPI_STORE, true>,
                                    mA, mB, mC, mW, p);
    if (e != cudaSuccess) return FP8FG_ERR_CUDA;
  }
  if (plan.sk_tiles > 0) {
    const dim3 fgrid(static_cast<unsigned>(plan.sk_tiles), kFixupCtasPerTile);
    if (p.c_f32)
      streamk_fixup_kernel<true><<<fgrid, kFixupThreads, 0, st>>>(static_cast<const float*>(ws), c, p);
    else
      streamk_fixup_kernel<false><<<fgrid, kFixupThreads, 0, st>>>(static_cast<const float*>(ws), c, p);
    if (cudaGetLastError() != cudaSuccess) return FP8FG_ERR_CUDA;
  }
  return FP8FG_OK;
}

fp8fg_status launch_gemm_quant(const uint8_t* a, const float* sa, const uint8_t* b,
                               const float* sb, uint8_t* q, float* s, int64_t M, int64_t N,
                               int64_t K, bool b_tile, bool pow2, cudaStream_t st) {
  CUtensorMap mA, mB, mQ;
  if (!make_maps(&mA, &mB, a, M, b, 0, N, K)) return FP8FG_ERR_CUDA;
  // codes [M, N] stored by 32-row x 64-byte boxes from 64-byte-swizzled staging
  const uint64_t dQ[2] = {static_cast<uint64_t>(N), static_cast<uint64_t>(M)};
  const uint64_t sQ[1] = {static_cast<uint64_t>(N)};
  const uint32_t boxQ[2] = {CST_ROW, 32};
  if (!encode_tensor_map(&mQ, CU_TENSOR_MAP_DATA_TYPE_UINT8, q, 2, dQ, sQ, boxQ,
                         CU_TENSOR_MAP_SWIZZLE_64B))
    return FP8FG_ERR_CUDA;
  if ((b_tile ? set_smem_attr<false, true, EPI_QUANT>() : set_smem_attr<false, false, EPI_QUANT>()) !=
      cudaSuccess)
    return FP8FG_ERR_CUDA;
  GemmParams p{};
  p.sa = sa;
  p.sb = sb;
  p.c = q;
  p.offsets = nullptr;
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.nkb = static_cast<int>(K / BK);
  p.m_tiles = static_cast<int>((M + BM - 1) / BM);
  p.n_tiles = static_cast<int>((N + BN - 1) / BN);
  p.group_m = group_m_tiles(p.m_tiles, K);
  p.E = 1;
  p.c_f32 = 0;
  p.b_tile = b_tile ? 1 : 0;
  p.s_out = s;
  p.pow2_out = pow2 ? 1 : 0;
  p.wait_limit = wait_limit_cycles();
  p.status = device_status_word();
  const int tiles = p.m_tiles * p.n_tiles;
  const int grid = tiles < device_sm_count() ? tiles : device_sm_count();
  if (b_tile)
    blockscaled_gemm_kernel<false, true, EPI_QUANT><<<grid, NUM_THREADS, smem_bytes<false, true>(), st>>>(mA, mB, mQ, mQ, p);
  else
    blockscaled_gemm_kernel<false, false, EPI_QUANT><<<grid, NUM_THREADS, smem_bytes<false, false>(), st>>>(mA, mB, mQ, mQ, p);
  return cudaGetLastError() == cudaSuccess ? FP8FG_OK : FP8FG_ERR_CUDA;
}

fp8fg_status launch_grouped_gemm(const uint8_t* a, const float* sa, const int32_t* offsets,
                                 int32_t E, int64_t total_rows, const uint8_t* b, const float* sb,
                                 void* c, fp8fg_dtype ct, int64_t N, int64_t K, cudaStream_t st) {
  CUtensorMap mA, mB, mC;
  // an empty A (no rows) still needs valid maps: point them at one row
  const int64_t map_rows = total_rows > 0 ? total_rows : 1;
  if (!make_maps(&mA, &mB, a, map_rows, b, E, N, K) || !make_c_map(&mC, c, ct, map_rows, N))
    return FP8FG_ERR_CUDA;
  if (set_smem_attr<true, false>() != cudaSuccess) return FP8FG_ERR_CUDA;
  GemmParams p{};
  p.sa = sa;
  p.sb = sb;
  p.c = c;
  p.offsets = offsets;
  p.M = static_cast<int>(total_rows);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.nkb = static_cast<int>(K / BK);
  p.m_tiles = 0;
  p.n_tiles = static_cast<int>((N + BN - 1) / BN);
  p.E = E;
  p.c_f32 = ct == FP8FG_F32;
  p.b_tile = 0;
  p.wait_limit = wait_limit_cycles();
  p.status = device_status_word();
  blockscaled_gemm_kernel<true, false, EPI_STORE><<<device_sm_count(), NUM_THREADS, smem_bytes<true, false>(), st>>>(
      mA, mB, mC, mC, p);
  return cudaGetLastError() == cudaSuccess ? FP8FG_OK : FP8FG_ERR_CUDA;
}

fp8fg_status launch_grouped_swiglu_quant(const uint8_t* a, const float* sa,
                                         const int32_t* offsets, int32_t E, int64_t total_rows,
                                         const uint8_t* b, const float* sb, uint8_t* q, float* s,
                                         int64_t N, int64_t K, bool pow2, cudaStream_t st) {
  CUtensorMap mA, mB;
  if (!make_maps(&mA, &mB, a, total_rows > 0 ? total_rows : 1, b, E, N, K)) return FP8FG_ERR_CUDA;
  // B as a 5-D view of [E, N = 2I, K]: {K, 64 rows, gate/up (stride I rows),
  // 64-row block (stride 64 rows), expert}; a box of {128, 64, 2, 2, 1} is one
  // pipeline stage: gate and up rows of 128 outputs, 64 at a time
  {
    const uint64_t I = static_cast<uint64_t>(N / 2), Ku = static_cast<uint64_t>(K);
    const uint64_t dB[5] = {Ku, 64, 2, I / 64, static_cast<uint64_t>(E)};
    const uint64_t sB[4] = {Ku, I * Ku, 64 * Ku, 2 * I * Ku};
    const uint32_t boxB[5] = {BK, 64, 2, 2, 1};
    if (!encode_tensor_map_u8(&mB, b, 5, dB, sB, boxB)) return FP8FG_ERR_CUDA;
  }
  if (set_smem_attr<true, false, EPI_SWIGLU>() != cudaSuccess) return FP8FG_ERR_CUDA;
  GemmParams p{};
  p.sa = sa;
  p.sb = sb;
  p.c = q;
  p.offsets = offsets;
  p.M = static_cast<int>(total_rows);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.nkb = static_cast<int>(K / BK);
  p.m_tiles = 0;
  p.n_tiles = static_cast<int>(N / BN);       // one tile: 128 outputs = 128 gate + 128 up rows
  p.E = E;
  p.c_f32 = 0;
  p.b_tile = 0;
  p.s_out = s;
  p.pow2_out = pow2 ? 1 : 0;
  p.wait_limit = wait_limit_cycles();
  p.status = device_status_word();
  // h codes [total_rows, N/2] stored by 32-row x 64-byte boxes from swizzled staging
  CUtensorMap mQ;
  const uint64_t dQ[2] = {static_cast<uint64_t>(N / 2),
                          static_cast<uint64_t>(total_rows > 0 ? total_rows : 1)};
  const uint64_t sQ[1] = {static_cast<uint64_t>(N / 2)};
  const uint32_t boxQ[2] = {CST_ROW, 32};
  if (!encode_tensor_map(&mQ, CU_TENSOR_MAP_DATA_TYPE_UINT8, q, 2, dQ, sQ, boxQ,
                         CU_TENSOR_MAP_SWIZZLE_64B))
    return FP8FG_ERR_CUDA;
  blockscaled_gemm_kernel<true, false, EPI_SWIGLU><<<device_sm_count(), NUM_THREADS, smem_bytes<true, false>(),
                                                     st>>>(mA, mB, mQ, mQ, p);
  return cudaGetLastError() == cudaSuccess ? FP8FG_OK : FP8FG_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// Allocation-free variant of the stream-K GEMM.  Some callers cannot allocate
// device memory when they call the GEMM (code that runs while a memory pool is
// locked or being captured, allocators that must not be re-entered, embedded
// runtimes with a fixed memory budget).  For them the split's partial tiles go
// to this file-scope array instead of a caller workspace.  It holds the split
// of up to kNoAllocMaxSms SMs (128 KB each, 20 MiB); every GPU that loads the
// library keeps it until the process exits.
constexpr int kNoAllocMaxSms = 160;
constexpr size_t kNoAllocScratchBytes = static_cast<size_t>(kNoAllocMaxSms) * BM * BN * sizeof(float);
static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchBytes / sizeof(float)];

namespace {

// Device address of g_noalloc_scratch on the current device, looked up on the
// first call on each device (host code cannot use the symbol itself: it names a
// host-side stand-in, not device memory).
float* noalloc_scratch_address() {
  static std::atomic<float*> cache[kMaxDevices] = {};
  const int d = current_device();
  if (d < 0) return nullptr;
  float* p = cache[d].load(std::memory_order_acquire);
  if (p != nullptr) return p;
  void* addr = nullptr;
  if (cudaGetSymbolAddress(&addr, g_noalloc_scratch) != cudaSuccess || addr == nullptr)
    return nullptr;
  p = static_cast<float*>(addr);
  cache[d].store(p, std::memory_order_release);
  return p;
}

}  // namespace

fp8fg_status launch_gemm_noalloc(const uint8_t* a, const float* sa, const uint8_t* b,
                                 const float* sb, void* c, fp8fg_dtype ct, int64_t M, int64_t N,
                                 int64_t K, bool b_tile, bool force_sk, cudaStream_t st) {
  if (gemm_workspace_bytes(M, N, K, false, force_sk) > kNoAllocScratchBytes)
    return FP8FG_ERR_UNSUPPORTED_SHAPE;      // the split on this device needs more than the array
  float* scratch = noalloc_scratch_address();
  if (scratch == nullptr) return FP8FG_ERR_CUDA;
  return launch_gemm(a, sa, b, sb, c, ct, M, N, K, b_tile, false, scratch, kNoAllocScratchBytes,
                     force_sk, st);
}

cudaError_t launch_wait_timeout_selftest(uint32_t limit_cycles, cudaStream_t st) {
  wait_timeout_selftest_kernel<<<1, 32, 0, st>>>(static_cast<long long>(limit_cycles),
                                                 device_status_word());
  return cudaGetLastError();
}

}  // namespace fp8fg
