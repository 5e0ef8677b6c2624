// Factored DoRA row norm on GB300 (sm_103a): tcgen05 tensor-core GEMMs fed by
// TMA, accumulating in tensor memory.
//
// Method source: web page "人工智能训练新突破：Anthropic团队破解大模型微调内存瓶颈难题"
// (techwalker.com), paragraph on factored normalisation: the row norm of
// W0 + s B A splits into a base, a cross and a Gram term, so memory falls from
// O(out*in) to O(out*r + r^2).  Written out,
//     n_i^2 = ||W0_i||^2 + 2 s <U_i, B_i> + s^2 B_i G B_i^T,  U = W0 A^T,  G = A A^T.
// The cross and Gram terms are folded into ONE accumulator per output row:
//     D_i = W0_i A^T + B_i (s/2 G)            (K = in + r)
//     n_i^2 = ||W0_i||^2 + 2 s <B_i, D_i>
// so U never reaches global memory; only G (r x r) does.
//
// Launch sequence of dora_norm_factored (the forward norm):
//   1. split_hl_kernel   A -> bf16 (A_h, A_l), the split N operand (see
//                        Precision); zeroes the launch's counters
//   2. fwd_norm_kernel   one cooperative launch: the Gram pieces of G = A A^T,
//                        their reduction into s/2 G (split like A), and the
//                        norm GEMM [W0 | B] x [A | s/2 G]^T whose epilogue
//                        reduces each row to (sum W0_i^2 over its K range,
//                        <B_i, D_i>); the epilogue warp that writes the last
//                        records of a quarter M tile sums them in a fixed
//                        order and writes n = sqrt(max(0, n^2)) and g = m / n
// (structure and work split: see the comment above fwd_norm_kernel)
//
// Precision of the forward norm: every fp32 operand is split x = h + l,
// h = bf16(x) and l = bf16(x - h) (nearest even; x - h is exact in fp32, so
// |x - h - l| <= 2^-18 |x|).  Each product is three kind::f16 MMAs on bf16
// operands,
//     x*y ~ h_x*h_y + l_x*h_y + h_x*l_y
// with fp32 accumulation in tensor memory; every bf16 x bf16 product is exact
// in fp32, and the dropped l_x*l_y and residual terms are <= 3 * 2^-18 of the
// product.  The M-side operand (W0, B or A) is split by converter warps, which
// read the raw box from shared memory, accumulate ||W0_i||^2 on the way and
// write h and l into tensor memory, where the MMAs take their A operand; the
// N-side operand (A, re-read by every M tile, and s/2 G) is split once in
// global memory.
//
// The gradient through the norm (dora_norm_factored_bwd) runs the same
// scheme in tc_gemm_kernel for its two large products (dB and dA, each one
// pass over W0).  Its first launch, grad_prep_kernel, splits the passes' N
// operands and, for r <= kSgMaxR, forms the Gram products G and s H on the
// CUDA cores as fp32 partials that sg_fin_kernel sums; for larger r those are
// two more tc_gemm_kernel passes with their reductions.
//
// tc_gemm structure (one CTA per SM, persistent, 192 threads):
//   warp 0      TMA producer: loads the raw M-side box [128 x 32 fp32] and the
//               N-side h / l boxes [NC x 32 bf16] of each K block into a ring
//               of stages
//   warp 1      allocates tensor memory; one lane issues tcgen05.mma
//   warps 2..5  converters (h / l split of the M-side box into the stage's
//               tensor-memory slot), then the epilogue for their 32
//               tensor-memory lanes each
// Tiles in shared memory are K-major with the swizzle of one K block per row:
// the raw fp32 box 128-byte rows (128-byte swizzle), the bf16 N-side boxes
// 64-byte rows (64-byte swizzle).  Tensor memory holds the accumulator and one
// operand slot per stage.  The work is the list of (M tile, N chunk, K block)
// units, split evenly over the CTAs; a CTA's range crosses at most a few tile
// boundaries, and each piece ("segment") leaves one partial result.  All
// partial sums are combined in a fixed order, so results are bitwise
// reproducible.
//
// Every wait on a shared-memory barrier (and, in fwd_norm_kernel, on a global
// counter) is bounded (kWaitLimitNs).  A wait that gives up sets a CTA abort
// flag, records a code in a device error word and makes all roles leave their
// loops; the producers then wait (bounded) for their copies in flight, the
// MMA lane for its issued MMAs, and tensor memory is freed before the CTA
// exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace {

constexpr int kBM = 128;            // rows per M tile (= tensor-memory lanes)
// K indices per K block of tc_gemm_kernel: one 128-byte fp32 row of the raw
// M-side box (TMA streams a large matrix from HBM faster through 128-byte box
// rows than through 64-byte ones: measured 4.5 vs 3.8 TB/s on GB300)
constexpr int kBK = 32;
constexpr int kThreads = 192;
constexpr int kMaxChunkN = 384;     // largest N handled by one CTA pass
constexpr int kMaxR = 1024;
constexpr int kMaxCtas = 160;       // CTAs of a launch at most (GB300 has 152 SMs); bounds the workspace
constexpr int kMinUnitsNorm = 4;
constexpr int kMinUnitsGram = 16;
constexpr int kSmemMax = 232448;           // 227 KB: the opt-in maximum per CTA
constexpr int kMaxStages = 12;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s
// ROWS passes: K indices per accumulation window.  The tensor core's fp32
// accumulation rounds toward zero, so its error grows with the length of an
// accumulation chain; windows of 1024 K summed in round-to-nearest keep the
// gradient's error near that of a plain fp32 loop.
constexpr int kChainK = 1024;

// kGram: partial tiles of a symmetric product (upper triangle only);
// kNorm: per-row <B_i, D_i> records and the fused n / g finalize (the forward
//        norm kernels: fwd_norm_kernel, tc16_kernel);
// kRows: partial rows of a plain product per CTA part, summed by rows_reduce_kernel
//        (tc_gemm_kernel, with kGram, for the gradient through the norm)
enum Mode : int { kGram = 0, kNorm = 1, kRows = 2 };

// device error word: 0 = fine; otherwise the code of the wait that gave up
__device__ int g_dora_err = 0;
// test hook (dora_test_stall_loads): the GEMM producers withhold all loads, so
// the other roles' bounded waits expire; and the limit of those waits
__device__ int g_dora_stall = 0;
__device__ unsigned long long g_wait_limit_ns = kWaitLimitNs;

struct TcParams {
  int mode;
  int M;            // valid M-side rows (out, or r for the Gram pass)
  int kb1;          // K blocks in segment 1 (W0 or A columns)
  int kbtot;        // K blocks in total (segment 2 = B / Gs columns)
  int nchunks;      // N chunks per M tile
  int sym;          // Gram pass: only tiles with N chunk >= M tile (G is symmetric; both 128 wide)
  int NC;           // N per chunk (multiple of 16, <= kMaxChunkN)
  int nbox;         // rows per N-side TMA box
  int nb;           // N-side boxes per stage (per h / l operand)
  int NT;           // N-side rows in shared memory per stage (nb * nbox >= NC)
  int nmma0, nmma1; // N of the first / second MMA instruction of a chunk
  // NT <= 128 (ROWS passes): h_x h_y and h_x l_y as one MMA of N = 2 NT over
  // the stage's h and l rows together (accumulator columns [0, NT) and
  // [NT, 2 NT), added in the epilogue): tc_gemm_kernel<XT, true>
  int dbl;
  int tmem_cols;
  int slot0;        // first tensor-memory column of the M-side operand slots (one slot per stage)
  int stages;
  int tiles;        // M tiles * nchunks (Gram pass: the upper-triangular tiles)
  long long units;  // tiles * kbtot
  int ctas;         // CTAs of the launch (one per SM at most)
  int ncl;          // = ctas: the parts the unit list is cut into
  int maxseg;
  unsigned stage_bytes;
  unsigned tx_bytes;
  float *part;      // GRAM: [tiles][maxseg][128][NC]; ROWS: [tiles][maxseg][NC / 4][128] float4
  int r;
  int *err;
  // ROWS: K blocks per accumulation window (the tensor-memory accumulator
  // restarts at every window boundary of the tile's K range, and each window
  // is added in fp32 round-to-nearest into the CTA's partial rows)
  int chain;
};

// c_i = (dL/dn_i) / n_i for a loss that sees n through g = m / n, with d_mag =
// dL/dm: dL/dn_i = -g_i d_mag_i
__device__ __forceinline__ float norm_grad_coef(const float *g, const float *d_mag, const float *norm, long long i) {
  return -(g[i] * d_mag[i]) / norm[i];
}

// K-block range [kb0, kbe) of the piece that starts at unit u of a CTA range
// ending at u_end: it ends at the tile's end, the range's end or (chain > 0)
// the next accumulation-window boundary
__device__ __forceinline__ int piece_end(long long u, long long u_end, int kb0, int kbtot, int chain) {
  int kbe = static_cast<int>(min(static_cast<long long>(kbtot), kb0 + (u_end - u)));
  if (chain > 0) kbe = min(kbe, (kb0 / chain + 1) * chain);
  return kbe;
}

// CTA that owns work unit u when `units` are split evenly over `ctas`.
__host__ __device__ __forceinline__ long long unit_begin(long long c, long long units, long long ctas) {
  return c * units / ctas;
}
__host__ __device__ __forceinline__ int cta_of(long long u, long long units, int ctas) {
  long long c = (u * ctas) / units;
  if (c >= ctas) c = ctas - 1;
  while (c + 1 < ctas && unit_begin(c + 1, units, ctas) <= u) ++c;
  while (c > 0 && unit_begin(c, units, ctas) > u) --c;
  return static_cast<int>(c);
}

// (M tile, N chunk) of work tile t.  Gram pass: the upper-triangular tiles
// (nc >= mt) of a q x q grid, row by row.  Norm pass: M tile t / nchunks,
// N chunk t % nchunks.
__host__ __device__ __forceinline__ void tile_coords(int t, int nchunks, int sym, int *mt, int *nc) {
  if (sym) {
    int i = 0;
    while (t >= nchunks - i) {
      t -= nchunks - i;
      ++i;
    }
    *mt = i;
    *nc = i + t;
  } else {
    *mt = t / nchunks;
    *nc = t - *mt * nchunks;
  }
}

// bounded wait whose limit (g_wait_limit_ns, a test hook) is read only on the
// slow path, so the common case -- the phase already complete -- touches no
// global memory
__device__ bool wait_bounded(uint32_t bar, uint32_t parity, SharedCtl *ctl, int *err, int code) {
  if (mbar_try_wait(bar, parity)) return true;
  return wait_bounded_ns(bar, parity, ctl, err, code, *reinterpret_cast<volatile unsigned long long *>(&g_wait_limit_ns));
}

// wait used while leaving after an abort: ignores the abort flag
__device__ void wait_drain(uint32_t bar, uint32_t parity) { wait_drain_ns(bar, parity, kWaitLimitNs); }

// ---------------------------------------------------------------------------
// the tensor-core GEMM of the gradient passes (GRAM or ROWS mode)
//
// XT: the M-side operand is stored K-major-transposed in global memory (its
// rows are K indices, its columns M indices, as W0 is for W0^T): the producer
// loads an unswizzled [BK x 128] box and the converters read it column-wise
// (lane = M row, conflict-free), the rest is unchanged.
// ---------------------------------------------------------------------------
// BKT: K indices per K block, 32 (one 128-byte fp32 box row) or 64 (two
// 128-byte-swizzled boxes side by side; XT: a [64 x 128] box), with N-side
// rows of 64 or 128 bytes
template <bool XT, bool DBL = false, int BKT = kBK>
__global__ void __launch_bounds__(kThreads, 1)
tc_gemm_kernel(const __grid_constant__ CUtensorMap mX1, const __grid_constant__ CUtensorMap mX2,
               const __grid_constant__ CUtensorMap mY1h, const __grid_constant__ CUtensorMap mY1l,
               const __grid_constant__ CUtensorMap mY2h, const __grid_constant__ CUtensorMap mY2l,
               const TcParams p) {
  constexpr int BK = BKT;
  static_assert(BK == 32 || BK == 64, "K blocks of 32 or 64");
  constexpr int kRowBytes = BK * 4;    // the raw fp32 M-side block's row (XT: column)
  constexpr int kBoxBytes = kBM * 128; // one 128-byte-swizzled raw box [128 rows x 32 fp32]
  constexpr int kNRowBytes = BK * 2;   // one N-side row of BK bf16 (h or l)
  constexpr int kSlotCols = BK;        // tensor-memory columns of one M-side operand slot (h, then l)
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int S = p.stages;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + static_cast<size_t>(S) * p.stage_bytes);
  // barrier layout: full[S], conv[S], empty[S], accf, acce, fin
  SharedCtl *ctl = reinterpret_cast<SharedCtl *>(bars + 3 * S + 3);
  const uint32_t full0 = smem_u32(bars);
  const uint32_t conv0 = full0 + 8u * S;
  const uint32_t empty0 = conv0 + 8u * S;
  const uint32_t accf = empty0 + 8u * S;
  const uint32_t acce = accf + 8;
  const uint32_t fin = acce + 8;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full0 + 8u * s, 1);
      mbar_init(conv0 + 8u * s, 4);   // one arrival per converter warp
      mbar_init(empty0 + 8u * s, 1);
    }
    mbar_init(accf, 1);
    mbar_init(acce, 4);
    mbar_init(fin, 1);
    ctl->abort = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_map(&mX1);
    prefetch_map(&mY1h);
    prefetch_map(&mY1l);
    if (p.kbtot > p.kb1) {
      prefetch_map(&mX2);
      prefetch_map(&mY2h);
      prefetch_map(&mY2l);
    }
  }
  if (warp == 1) {
    __syncwarp();
    tmem_alloc(smem_u32(&ctl->tmem_base), static_cast<uint32_t>(p.tmem_cols));
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;

  const int cl = static_cast<int>(blockIdx.x);
  const long long u_begin = unit_begin(cl, p.units, p.ncl);
  const long long u_end = unit_begin(cl + 1, p.units, p.ncl);

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;  // loads issued in total (to drain on abort)
      bool ok = *reinterpret_cast<volatile int *>(&g_dora_stall) == 0;
      for (long long u = u_begin; u < u_end && ok;) {
        const int t = static_cast<int>(u / p.kbtot);
        const int kb0 = static_cast<int>(u - static_cast<long long>(t) * p.kbtot);
        const int kbe = piece_end(u, u_end, kb0, p.kbtot, p.chain);
        int mt, nc;
        tile_coords(t, p.nchunks, p.sym, &mt, &nc);
        for (int kb = kb0; kb < kbe; ++kb) {
          if (!wait_bounded(empty0 + 8u * stage, phase ^ 1u, ctl, p.err, 1)) {
            ok = false;
            break;
          }
          const uint32_t fb = full0 + 8u * stage;
          mbar_expect_tx(fb, p.tx_bytes);
          const uint32_t xs = smem_u32(smem + static_cast<size_t>(stage) * p.stage_bytes);
          const uint32_t yh = xs + kBM * kRowBytes;
          const uint32_t yl = yh + static_cast<uint32_t>(p.NT) * kNRowBytes;
          const bool seg1 = kb < p.kb1;
          const int kx = (seg1 ? kb : kb - p.kb1) * BK;    // first K index of the block
          if (XT) {
            tma_load_2d(xs, seg1 ? &mX1 : &mX2, mt * kBM, kx, fb);
          } else {
#pragma unroll
            for (int bx = 0; bx < BK / 32; ++bx)
              tma_load_2d(xs + bx * kBoxBytes, seg1 ? &mX1 : &mX2, kx + 32 * bx, mt * kBM, fb);
          }
          // the N-side tile of the chunk: the bf16 h and l operands
          for (int i = 0; i < p.nb; ++i) {
            const int ro = i * p.nbox;
            const int ny = nc * p.NC + ro;
            const uint32_t off = static_cast<uint32_t>(ro * kNRowBytes);
            tma_load_2d(yh + off, seg1 ? &mY1h : &mY2h, kx, ny, fb);
            tma_load_2d(yl + off, seg1 ? &mY1l : &mY2l, kx, ny, fb);
          }
          ++issued;
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        u += kbe - kb0;
      }
      if (!ok) {
        // drain: the last min(issued, S) stages may still have copies in flight
        int st = stage;
        uint32_t ph = phase;
        for (int k = 0; k < S && k < issued; ++k) {
          if (--st < 0) {
            st = S - 1;
            ph ^= 1u;
          }
          wait_drain(full0 + 8u * st, ph);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      int stage = 0;
      uint32_t phase = 0;
      uint32_t aphase = 0;
      bool ok = true;
      const uint32_t ic0 = idesc_bf16(p.nmma0);
      const uint32_t ic1 = p.nmma1 > 0 ? idesc_bf16(p.nmma1) : 0u;
      const uint32_t icd = DBL ? idesc_bf16(2 * p.NT) : 0u;
      for (long long u = u_begin; u < u_end && ok;) {
        const int t = static_cast<int>(u / p.kbtot);
        const int kb0 = static_cast<int>(u - static_cast<long long>(t) * p.kbtot);
        const int kbe = piece_end(u, u_end, kb0, p.kbtot, p.chain);
        if (!wait_bounded(acce, aphase ^ 1u, ctl, p.err, 3)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int kb = kb0; kb < kbe; ++kb) {
          if (!wait_bounded(conv0 + 8u * stage, phase, ctl, p.err, 2)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t yh = smem_u32(smem + static_cast<size_t>(stage) * p.stage_bytes) + kBM * kRowBytes;
          const uint32_t yl = yh + static_cast<uint32_t>(p.NT) * kNRowBytes;
          // M-side operand slot: BK/2 columns of h (two bf16 per column,
          // K-consecutive), then BK/2 columns of l.  Per K = 16 step three
          // products h_x h_y + l_x h_y + h_x l_y into the same accumulator.
          const uint32_t sh = tmem + static_cast<uint32_t>(p.slot0 + stage * kSlotCols);
          const uint32_t sl = sh + BK / 2;
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            const uint32_t acc0 = (kb != kb0 || k != 0) ? 1u : 0u;
            const uint32_t ko = static_cast<uint32_t>(k) * 32u;   // 16 bf16 along the 64-byte row
            const uint32_t ah = sh + 8u * k, al = sl + 8u * k;
            {
              const uint64_t bh = sdesc<BK / 2>(yh + ko), bl = sdesc<BK / 2>(yl + ko);
              if constexpr (DBL) {
                mma_bf16_ta(tmem, ah, bh, icd, acc0);   // rows [h; l] of the stage: h_x h_y | h_x l_y
                mma_bf16_ta(tmem, al, bh, ic0, 1u);
                (void)bl;
              } else {
                mma_bf16_ta(tmem, ah, bh, ic0, acc0);
                mma_bf16_ta(tmem, al, bh, ic0, 1u);
                mma_bf16_ta(tmem, ah, bl, ic0, 1u);
              }
            }
            if (p.nmma1 > 0) {
              const uint32_t no = 256u * kNRowBytes;
              const uint64_t bh = sdesc<BK / 2>(yh + no + ko), bl = sdesc<BK / 2>(yl + no + ko);
              mma_bf16_ta(tmem + 256u, ah, bh, ic1, acc0);
              mma_bf16_ta(tmem + 256u, al, bh, ic1, 1u);
              mma_bf16_ta(tmem + 256u, ah, bl, ic1, 1u);
            }
          }
          mma_commit(empty0 + 8u * stage);
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(accf);
        aphase ^= 1u;
        u += kbe - kb0;
      }
      // all issued MMAs must finish before tensor memory is released
      mma_commit(fin);
      wait_drain(fin, 0);
    }
  } else {
    // -------------------------------------------------------- converters + epilogue
    const int quad = warp & 3;            // tensor-memory lane group of this warp
    const int row = quad * 32 + lane;     // row within the M tile
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    // accumulator columns [c, c + 32) of this warp's rows; with DBL the
    // h_x l_y half (NT columns on) is added in
    const int nt_cols = p.NT;
    auto acc_ld32 = [&](int c, float (&v)[32]) {
      tmem_ld32(lane_addr + static_cast<uint32_t>(c), v);
      if constexpr (DBL) {
        float w[32];
        tmem_ld32(lane_addr + static_cast<uint32_t>(nt_cols + c), w);
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] += w[e];
      }
    };
    int stage = 0;
    uint32_t phase = 0;
    uint32_t aphase = 0;
    bool ok = true;
    for (long long u = u_begin; u < u_end && ok;) {
      const int t = static_cast<int>(u / p.kbtot);
      const int kb0 = static_cast<int>(u - static_cast<long long>(t) * p.kbtot);
      const int kbe = piece_end(u, u_end, kb0, p.kbtot, p.chain);
      int mt, nc;
      tile_coords(t, p.nchunks, p.sym, &mt, &nc);
      const size_t tm = static_cast<size_t>(mt) * p.nchunks + nc;   // (M tile, N chunk) of this CTA's partials
      for (int kb = kb0; kb < kbe; ++kb) {
        // every lane waits; the decision to go on is taken warp-wide so that
        // the warp stays converged for the tcgen05.ld of the epilogue
        const bool got = wait_bounded(full0 + 8u * stage, phase, ctl, p.err, 4);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        // this thread's row: BK fp32 in BK/4 16-byte chunks, stored swizzled
        // (swz_chunk); one K = 16 step at a time, split into the stage's
        // tensor-memory operand slot: 8 columns of h pairs and 8 of l pairs
        const uint8_t *xbox = smem + static_cast<size_t>(stage) * p.stage_bytes;
        const float4 *xr = reinterpret_cast<const float4 *>(xbox + row * 128);   // row `row` of raw box 0
        const float *xc = reinterpret_cast<const float *>(xbox) + row;   // XT: column `row` of [BK][128]
        const uint32_t slot = lane_addr + static_cast<uint32_t>(p.slot0 + stage * kSlotCols);
        auto load8 = [&](int q, float (&v)[8]) {
          if (XT) {
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = xc[(8 * q + e) * kBM];
          } else {
            // K indices 8q .. 8q + 7: chunks 2q, 2q + 1 of raw box q / 4
            const float4 *xq = xr + (q >> 2) * (kBoxBytes / 16);
            const float4 a = xq[swz_chunk<32>((2 * q) & 7, row)], b = xq[swz_chunk<32>((2 * q + 1) & 7, row)];
            v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
            v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
          }
        };
        // x = h + l: h = bf16(x), l = bf16(x - h); column c of a step holds
        // the K indices 2c, 2c + 1
#pragma unroll
        for (int q16 = 0; q16 < BK / 16; ++q16) {
          uint32_t hb[8], lb[8];
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            float v[8];
            load8(2 * q16 + half, v);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float x0 = v[2 * e], x1 = v[2 * e + 1];
              const uint32_t h = pack_bf16x2(x0, x1);
              hb[4 * half + e] = h;
              lb[4 * half + e] =
                  pack_bf16x2(x0 - __uint_as_float(h << 16), x1 - __uint_as_float(h & 0xffff0000u));
            }
          }
          tmem_st8(slot + 8u * q16, hb);
          tmem_st8(slot + BK / 2 + 8u * q16, lb);
        }
        tmem_wait_st();
        // the tensor-memory stores are complete (wait::st); order them before
        // the MMA lane's work, then one arrival per warp
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(conv0 + 8u * stage);
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      const int grow = mt * kBM + row;
      const bool valid = grow < p.M;
      const int seg = cl - cta_of(static_cast<long long>(t) * p.kbtot, p.units, p.ncl);
      // ---- epilogue of this segment
      const bool got = wait_bounded(accf, aphase, ctl, p.err, 5);
      if (!__all_sync(0xffffffffu, got)) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (p.mode == kGram) {
        float *dst = p.part + ((tm * p.maxseg + seg) * kBM + row) * p.NC;
        for (int c = 0; c < p.NC; c += 32) {
          float v[32];
          acc_ld32(c, v);
          if (valid) {
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
              if (c + j < p.NC) *reinterpret_cast<float4 *>(dst + c + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
            }
          }
        }
      } else {
        // ROWS.  The CTA part's partial rows, [NC/4 column groups][128 rows]
        // of float4 (a warp's store covers 32 consecutive rows: 512 bytes).
        // The part's first window stores; later windows add in fp32 with
        // fire-and-forget reductions (one thread per address, in program
        // order, so the sum order is fixed).  rows_reduce_kernel sums the parts.
        const bool first = u == u_begin || kb0 == 0;
        const size_t slot_f4 = static_cast<size_t>(32) * p.NC;   // float4s per partial slot
        float4 *mine = reinterpret_cast<float4 *>(p.part) + (tm * p.maxseg + seg) * slot_f4 + row;
        for (int c = 0; c < p.NC; c += 32) {
          float v[32];
          acc_ld32(c, v);
          if (valid) {
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              if (c + 4 * q < p.NC) {
                float4 *dst = mine + static_cast<size_t>(c / 4 + q) * kBM;
                if (first) *dst = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
                else red_add_f32x4(dst, v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
              }
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acce);
      aphase ^= 1u;
      u += kbe - kb0;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem, static_cast<uint32_t>(p.tmem_cols));
  }
}

// ---------------------------------------------------------------------------
// the forward norm in one launch, bf16 three-product scheme
//
// CTAs are one per SM and all co-resident (cooperative launch).
//   Gram phase   CTAs 0 .. g-1 only: each upper-triangular tile of G = A A^T
//                (M side A raw, N side A split) is cut along K into P pieces,
//                one per CTA, each written as a partial tile;
//   reduction    the P CTAs of a tile wait for one another's pieces (a
//                per-tile counter), then each reduces its share of the tile's
//                32 x 32 blocks of s/2 G: the P pieces of each entry summed in
//                a fixed order, scaled, split into bf16 h and l, written with
//                the mirror entry;
//   norm phase   every CTA: its share of the (M tile, K block) units of
//                [W0 | B] x [A | s/2 G]^T with the fused per-row epilogue and
//                n / g finalize.  The split is weighted: the Gram CTAs take
//                fewer units, so that all CTAs finish together.  A CTA takes
//                its segments last first, so it reaches an s/2 G tail only
//                after most of its W0 work; the N-side producer's first tail
//                load waits for every reduction to be complete (a grid-wide
//                counter), which by then it always is.
// The raw M-side boxes have a ring of their own, released by the converter
// warps as soon as they have split a box into tensor memory; the N-side tiles
// and the tensor-memory operand slots share a second ring, released by the
// MMAs.  The rings run on across the two phases, so the producers already
// fetch the norm phase's W0 while the converter warps reduce G.
//
//   warp 0      lane 0: TMA producer of the raw M-side boxes [128 x 32 fp32]
//   warp 1      allocates tensor memory; lane 0 issues the MMAs
//   warps 2..5  converters (split into tensor memory, row sums of W0^2), the
//               epilogues of their 32 tensor-memory lanes, the reduction
//   warp 6      lane 0: TMA producer of the N-side h and l tiles [NT x 32 bf16]
// ---------------------------------------------------------------------------
constexpr int kFwdThreads = 224;
// K indices per K block of fwd_norm_kernel<FBK>: 32, or 64 where the
// accumulator leaves tensor memory for at least four 64-column operand slots
// (N <= 256): half the barrier waits and slot releases per W0 byte
constexpr int kFwdBox = 32;                      // K indices of one raw M-side box (128-byte rows)
constexpr int kFwdBoxBytes = kBM * kFwdBox * 4;  // 16 KB
constexpr int kFwdMaxX = 16;
constexpr int kFwdMaxS = 8;
constexpr int kGramPieces = 8;                   // CTAs (K pieces) per Gram tile, at most (16 was 3-4% slower at r = 256)

// one phase's work list and N-side geometry
struct FwdPhase {
  int kb1, kbtot;   // K blocks of the first operand pair / in total
  int nchunks, sym, NC;
  int nbox, nb;     // N-side rows per TMA box, boxes per tile
  int nmma0, nmma1; // N of the accumulator's two MMA instructions (nmma1 = 0: one)
  int tiles;
  long long units;  // tiles * kbtot
  int ctas;         // CTAs the units are split over (the first ones of the grid)
  int P;            // Gram phase: pieces per tile (CTA c < P * tiles takes piece c % P of tile c / P)
  float *part;      // Gram: [g][128][NC], the piece of CTA c at c;
                    // norm: [tiles + ctas][128] float2, the records of tile t
                    // from CTA c at t + c (CTAs touch tiles in ascending
                    // order, so t + c is unique)
};

struct FwdParams {
  FwdPhase ph[2];   // 0: Gram, 1: norm
  int fbk;          // K indices per K block (the kernel instance)
  int M;            // out (rows of the norm phase)
  int r, npad;
  int NT;           // N-side rows of a stage (the larger phase's)
  // NT <= 64: h_x h_y and h_x l_y as ONE MMA of N = 2 NT over the stage's h
  // and l rows together (accumulator columns [0, NT) and [NT, 2 NT), added in
  // the epilogue), then l_x h_y: two MMAs per K = 16 step instead of three
  int dbl;
  int tmem_cols, slot0;
  int S;            // N-side stages = tensor-memory operand slots
  int SX;           // raw M-side box slots
  unsigned y_bytes; // one N-side stage: the h tile then the l tile
  int ctas;
  int *err;
  int *cnt;         // norm: [M tiles][4] records written so far
  int *sync;        // [0] converter warps done reducing (4 per Gram CTA), [1 + t] those done with tile t's pieces
  int nsync;        // 1 + Gram tiles
  const float *m;
  float *norm, *g;
  float two_s, half_s;
  const float *Bk;
  int ldb;
  __nv_bfloat16 *gs_h, *gs_l;   // s/2 G split, [npad, npad] each
  int stage_b;      // the last epilogue stages B's rows through the operand rings (they are large enough)
  long long ub[kMaxCtas + 1];   // norm phase: CTA c takes units [ub[c], ub[c + 1]) (none empty)
};

// The CTA of the norm phase whose range holds unit u (ranges are non-empty
// and ascending: the largest c with ub[c] <= u)
__device__ __forceinline__ int split_cta_of(const long long *ub, int C, long long u) {
  int lo = 0, hi = C - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (ub[mid] <= u) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// The segments of a CTA's unit range [u_begin, hi) are taken last first: the
// one ending at hi is [max(u_begin, start of its tile), hi).  Returns its
// start (the next hi) and sets its tile and K-block range.  Taken in this
// order, a range that starts inside a tile's s/2 G tail reaches that tail
// last, long after the Gram reduction is complete.
__device__ __forceinline__ long long seg_range(long long u_begin, long long hi, int kbtot, int *t, int *kb0,
                                               int *kbe) {
  *t = static_cast<int>((hi - 1) / kbtot);
  const long long t0 = static_cast<long long>(*t) * kbtot;
  const long long lo = u_begin > t0 ? u_begin : t0;
  *kb0 = static_cast<int>(lo - t0);
  *kbe = static_cast<int>(hi - t0);
  return lo;
}

// This CTA's unit range in a phase: the Gram phase's fixed pieces (a tile's
// K blocks cut into P equal parts) or the norm phase's balanced split.
__device__ __forceinline__ void phase_range(const FwdParams &p, const FwdPhase &f, int c, long long *ub,
                                            long long *ue) {
  if (f.P > 0) {
    *ub = *ue = 0;
    if (c < f.P * f.tiles) {
      const int t = c / f.P, q = c - t * f.P;
      const long long t0 = static_cast<long long>(t) * f.kbtot;
      *ub = t0 + static_cast<long long>(q) * f.kbtot / f.P;
      *ue = t0 + static_cast<long long>(q + 1) * f.kbtot / f.P;
    }
  } else {
    *ub = p.ub[c];
    *ue = p.ub[c + 1];
  }
}

// global counter wait (ld.acquire), bounded like the barrier waits
__device__ __forceinline__ int ld_acquire(const int *p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ bool wait_count(const int *ctr, int target, SharedCtl *ctl, int *err, int code) {
  if (ld_acquire(ctr) >= target) return true;
  const unsigned long long t0 = globaltimer();
  const unsigned long long lim = *reinterpret_cast<volatile unsigned long long *>(&g_wait_limit_ns);
  for (;;) {
    __nanosleep(128);
    if (ld_acquire(ctr) >= target) return true;
    if (ctl->abort) return false;
    if (globaltimer() - t0 > lim) {
      ctl->abort = 1;
      atomicCAS(err, 0, code);
      return false;
    }
  }
}
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// s/2 G entry (a, b) split into bf16 h and l
__device__ __forceinline__ void store_gs3(__nv_bfloat16 *gh, __nv_bfloat16 *gl, int npad, int a, int b, float v) {
  const __nv_bfloat16 h = __float2bfloat16_rn(v);
  const long long i = static_cast<long long>(a) * npad + b;
  gh[i] = h;
  gl[i] = __float2bfloat16_rn(v - __bfloat162float(h));
}

// DBL: the plan's dbl (two MMAs per K = 16 step, N-side rows <= 64), a
// separate instance so that the other ranks' code is unchanged
template <int FBK, bool DBL = false>
__global__ void __launch_bounds__(kFwdThreads, 1)
fwd_norm_kernel(const __grid_constant__ CUtensorMap mA, const __grid_constant__ CUtensorMap mW0,
                const __grid_constant__ CUtensorMap mB, const __grid_constant__ CUtensorMap mAh_g,
                const __grid_constant__ CUtensorMap mAl_g, const __grid_constant__ CUtensorMap mAh_n,
                const __grid_constant__ CUtensorMap mAl_n, const __grid_constant__ CUtensorMap mGh,
                const __grid_constant__ CUtensorMap mGl, const __grid_constant__ CUtensorMap mBs,
                const FwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  static_assert(FBK == 32 || FBK == 64, "K blocks of 32 or 64");
  constexpr int kFwdBK = FBK;                        // K indices per K block
  constexpr int kXBoxes = FBK / kFwdBox;             // raw 32-wide boxes per raw-box slot
  constexpr int kFwdXBytes = kXBoxes * kFwdBoxBytes; // one raw-box slot
  constexpr int kFwdNRow = FBK * 2;                  // one N-side row of h or l (64 or 128 bytes)
  const int S = p.S, SX = p.SX;
  uint8_t *xring = smem;
  uint8_t *yring = smem + static_cast<size_t>(SX) * kFwdXBytes;
  uint64_t *bars = reinterpret_cast<uint64_t *>(yring + static_cast<size_t>(S) * p.y_bytes);
  // barrier layout: xfull[SX], xempty[SX], yfull[S], sfree[S], tconv[S], accf, acce, fin, stg[4]
  SharedCtl *ctl = reinterpret_cast<SharedCtl *>(bars + 2 * SX + 3 * S + 7);
  const uint32_t xfull0 = smem_u32(bars);
  const uint32_t xempty0 = xfull0 + 8u * SX;
  const uint32_t yfull0 = xempty0 + 8u * SX;
  const uint32_t sfree0 = yfull0 + 8u * S;
  const uint32_t tconv0 = sfree0 + 8u * S;
  const uint32_t accf = tconv0 + 8u * S;
  const uint32_t acce = accf + 8;
  const uint32_t fin = acce + 8;
  const uint32_t stg0 = fin + 8;   // one per converter warp: its rows of B, staged for the last epilogue

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < SX; ++i) {
      mbar_init(xfull0 + 8u * i, 1);
      mbar_init(xempty0 + 8u * i, 4);   // one arrival per converter warp
    }
    for (int i = 0; i < S; ++i) {
      mbar_init(yfull0 + 8u * i, 1);
      mbar_init(sfree0 + 8u * i, 1);    // the MMAs' commit
      mbar_init(tconv0 + 8u * i, 4);    // one arrival per converter warp
    }
    mbar_init(accf, 1);
    mbar_init(acce, 4);
    mbar_init(fin, 1);
    for (int i = 0; i < 4; ++i) mbar_init(stg0 + 8u * i, 1);
    ctl->abort = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_map(&mA);
    prefetch_map(&mW0);
    prefetch_map(&mB);
    prefetch_map(&mBs);
  }
  if (warp == 6 && lane == 0) {
    prefetch_map(&mAh_g);
    prefetch_map(&mAl_g);
    prefetch_map(&mAh_n);
    prefetch_map(&mAl_n);
    prefetch_map(&mGh);
    prefetch_map(&mGl);
  }
  if (warp == 1) {
    __syncwarp();
    tmem_alloc(smem_u32(&ctl->tmem_base), static_cast<uint32_t>(p.tmem_cols));
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  const int cl = static_cast<int>(blockIdx.x);

  if (warp == 0 || warp == 6) {
    if (lane == 0) {
      // ------------------------------------------- producers (M side / N side)
      const bool xside = warp == 0;
      const int R = xside ? SX : S;
      const uint32_t full0 = xside ? xfull0 : yfull0;
      const uint32_t free0 = xside ? xempty0 : sfree0;
      int slot = 0;
      uint32_t phase = 0;
      int issued = 0;
      bool ok = *reinterpret_cast<volatile int *>(&g_dora_stall) == 0;
      bool gs_ready = false;
      for (int ph = 0; ph < 2 && ok; ++ph) {
        const FwdPhase &f = p.ph[ph];
        long long u_begin, u_end;
        phase_range(p, f, cl, &u_begin, &u_end);
        // this CTA's segments, last first (see seg_range)
        for (long long hi = u_end; hi > u_begin && ok;) {
          int t, kb0, kbe;
          hi = seg_range(u_begin, hi, f.kbtot, &t, &kb0, &kbe);
          int mt, nc;
          tile_coords(t, f.nchunks, f.sym, &mt, &nc);
          for (int kb = kb0; kb < kbe; ++kb) {
            const bool seg1 = kb < f.kb1;
            if (!xside && ph == 1 && !seg1 && !gs_ready) {
              // the s/2 G tail: written by every CTA's reduction (generic
              // stores), read here by TMA
              if (!wait_count(p.sync + 0, 4 * p.ph[0].P * p.ph[0].tiles, ctl, p.err, 10)) {
                ok = false;
                break;
              }
              fence_proxy_async_global();
              gs_ready = true;
            }
            if (!wait_bounded(free0 + 8u * slot, phase ^ 1u, ctl, p.err, xside ? 1 : 6)) {
              ok = false;
              break;
            }
            const uint32_t fb = full0 + 8u * slot;
            const int kx = (seg1 ? kb : kb - f.kb1) * kFwdBK;
            if (xside) {
              mbar_expect_tx(fb, kFwdXBytes);
              const CUtensorMap *mx = ph == 0 ? &mA : (seg1 ? &mW0 : &mB);
#pragma unroll
              for (int b = 0; b < kXBoxes; ++b)
                tma_load_2d(smem_u32(xring + static_cast<size_t>(slot) * kFwdXBytes + b * kFwdBoxBytes), mx,
                            kx + kFwdBox * b, mt * kBM, fb);
            } else {
              const uint32_t ntile = static_cast<uint32_t>(f.nb * f.nbox) * kFwdNRow;
              mbar_expect_tx(fb, 2u * ntile);
              const uint32_t yh = smem_u32(yring + static_cast<size_t>(slot) * p.y_bytes);
              const uint32_t yl = yh + static_cast<uint32_t>(p.NT) * kFwdNRow;
              const CUtensorMap *mh = ph == 0 ? &mAh_g : (seg1 ? &mAh_n : &mGh);
              const CUtensorMap *ml = ph == 0 ? &mAl_g : (seg1 ? &mAl_n : &mGl);
              for (int i = 0; i < f.nb; ++i) {
                const int ro = i * f.nbox;
                const uint32_t off = static_cast<uint32_t>(ro * kFwdNRow);
                tma_load_2d(yh + off, mh, kx, nc * f.NC + ro, fb);
                tma_load_2d(yl + off, ml, kx, nc * f.NC + ro, fb);
              }
            }
            ++issued;
            if (++slot == R) {
              slot = 0;
              phase ^= 1u;
            }
          }
        }
      }
      if (!ok) {
        // drain: the last min(issued, R) slots may still have copies in flight
        int st = slot;
        uint32_t ph = phase;
        for (int k = 0; k < R && k < issued; ++k) {
          if (--st < 0) {
            st = R - 1;
            ph ^= 1u;
          }
          wait_drain(full0 + 8u * st, ph);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      int ss = 0;
      uint32_t sph = 0;
      uint32_t aphase = 0;
      bool ok = true;
      constexpr bool dbl = DBL;
      const uint32_t icd = dbl ? idesc_bf16(2 * p.NT) : 0u;
      for (int ph = 0; ph < 2 && ok; ++ph) {
        const FwdPhase &f = p.ph[ph];
        const uint32_t ic0 = idesc_bf16(f.nmma0);
        const uint32_t ic1 = f.nmma1 > 0 ? idesc_bf16(f.nmma1) : 0u;
        long long u_begin, u_end;
        phase_range(p, f, cl, &u_begin, &u_end);
        for (long long hi = u_end; hi > u_begin && ok;) {
          int t, kb0, kbe;
          hi = seg_range(u_begin, hi, f.kbtot, &t, &kb0, &kbe);
          if (!wait_bounded(acce, aphase ^ 1u, ctl, p.err, 3)) {
            ok = false;
            break;
          }
          tc_fence_after();
          for (int kb = kb0; kb < kbe; ++kb) {
            // the converters arrive once the slot is written AND its
            // N-side tile has landed: one barrier wait per K block here
            if (!wait_bounded(tconv0 + 8u * ss, sph, ctl, p.err, 2)) {
              ok = false;
              break;
            }
            tc_fence_after();
            // operand slot ss: 16 columns of h pairs, then 16 of l pairs; per
            // K = 16 step the products h_x h_y + l_x h_y + h_x l_y
            const uint32_t sh = tmem + static_cast<uint32_t>(p.slot0 + ss * kFwdBK);
            const uint32_t sl = sh + kFwdBK / 2;
            const uint32_t yh = smem_u32(yring + static_cast<size_t>(ss) * p.y_bytes);
            const uint32_t yl = yh + static_cast<uint32_t>(p.NT) * kFwdNRow;
#pragma unroll
            for (int k = 0; k < kFwdBK / 16; ++k) {
              const uint32_t acc0 = (kb != kb0 || k != 0) ? 1u : 0u;
              const uint32_t ko = static_cast<uint32_t>(k) * 32u;
              const uint32_t ah = sh + 8u * k, al = sl + 8u * k;
              {
                const uint64_t bh = sdesc<kFwdBK / 2>(yh + ko), bl = sdesc<kFwdBK / 2>(yl + ko);
                if constexpr (dbl) {
                  mma_bf16_ta(tmem, ah, bh, icd, acc0);   // rows [h; l] of the stage: h_x h_y | h_x l_y
                  mma_bf16_ta(tmem, al, bh, ic0, 1u);
                } else {
                  mma_bf16_ta(tmem, ah, bh, ic0, acc0);
                  mma_bf16_ta(tmem, al, bh, ic0, 1u);
                  mma_bf16_ta(tmem, ah, bl, ic0, 1u);
                }
              }
              if (f.nmma1 > 0) {
                const uint32_t no = 256u * kFwdNRow;
                const uint64_t bh = sdesc<kFwdBK / 2>(yh + no + ko), bl = sdesc<kFwdBK / 2>(yl + no + ko);
                mma_bf16_ta(tmem + 256u, ah, bh, ic1, acc0);
                mma_bf16_ta(tmem + 256u, al, bh, ic1, 1u);
                mma_bf16_ta(tmem + 256u, ah, bl, ic1, 1u);
              }
            }
            mma_commit(sfree0 + 8u * ss);
            if (++ss == S) {
              ss = 0;
              sph ^= 1u;
            }
          }
          if (!ok) break;
          mma_commit(accf);
          aphase ^= 1u;
        }
      }
      // all issued MMAs must finish before tensor memory is released
      mma_commit(fin);
      wait_drain(fin, 0);
    }
  } else {
    // ------------------------------------------- converters, epilogues, reduction
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const int ct = threadIdx.x - 64;   // 0..127 over the four converter warps
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    // accumulator columns [c, c + 32) of this warp's rows; with p.dbl the
    // h_x l_y half (NT columns on) is added in
    const int nt_cols = p.NT;
    auto acc_ld32 = [&](int c, float (&v)[32]) {
      tmem_ld32(lane_addr + static_cast<uint32_t>(c), v);
      if constexpr (DBL) {
        float w[32];
        tmem_ld32(lane_addr + static_cast<uint32_t>(nt_cols + c), w);
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] += w[e];
      }
    };
    int xs = 0, ss = 0;
    uint32_t xph = 0, sph = 0;
    uint32_t aphase = 0;
    bool ok = true;
    for (int ph = 0; ph < 2 && ok; ++ph) {
      const FwdPhase &f = p.ph[ph];
      const bool norm = ph == 1;
      long long u_begin, u_end;
      phase_range(p, f, cl, &u_begin, &u_end);
      for (long long hi = u_end; hi > u_begin && ok;) {
        int t, kb0, kbe;
        hi = seg_range(u_begin, hi, f.kbtot, &t, &kb0, &kbe);
        int mt, nc;
        tile_coords(t, f.nchunks, f.sym, &mt, &nc);
        const size_t tm = static_cast<size_t>(mt) * f.nchunks + nc;
        const int kpf = kbe - 8 > kb0 ? kbe - 8 : kb0;   // K block at which B's rows are prefetched
        float n0 = 0.0f;
        for (int kb = kb0; kb < kbe; ++kb) {
          if (norm && kb == kpf && lane == 0) {
            // the epilogue will read this warp's 32 rows of B: start them
            // towards L2 a few K blocks before the segment ends
            const int r0 = mt * kBM + quad * 32;
            const int nr = min(32, p.M - r0);
            if (nr > 0)
              prefetch_l2(p.Bk + static_cast<size_t>(r0) * p.ldb, static_cast<uint32_t>(nr) * p.ldb * 4u);
          }
          // the raw box has landed and the operand slot is free (its previous
          // MMAs are complete); the decision is warp-wide
          const bool got = wait_bounded(xfull0 + 8u * xs, xph, ctl, p.err, 4) &&
                           wait_bounded(sfree0 + 8u * ss, sph ^ 1u, ctl, p.err, 8);
          if (!__all_sync(0xffffffffu, got)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // row `row` of raw box b: 32 fp32 in 8 16-byte chunks, swizzled
          const uint8_t *xrow = xring + static_cast<size_t>(xs) * kFwdXBytes + row * (kFwdBox * 4);
          const uint32_t slot = lane_addr + static_cast<uint32_t>(p.slot0 + ss * kFwdBK);
          float blk = 0.0f;
#pragma unroll
          for (int q16 = 0; q16 < kFwdBK / 16; ++q16) {
            uint32_t hb[8], lb[8];
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              const int q = 2 * q16 + half;
              const float4 *xr = reinterpret_cast<const float4 *>(xrow + (q >> 2) * kFwdBoxBytes);
              const int qq = q & 3;   // group of 8 K within the box
              const float4 a = xr[swz_chunk<kFwdBox>(2 * qq, row)], b = xr[swz_chunk<kFwdBox>(2 * qq + 1, row)];
              const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float x0 = v[2 * e], x1 = v[2 * e + 1];
                blk = fmaf(x0, x0, blk);
                blk = fmaf(x1, x1, blk);
                const uint32_t h = pack_bf16x2(x0, x1);
                hb[4 * half + e] = h;
                lb[4 * half + e] =
                    pack_bf16x2(x0 - __uint_as_float(h << 16), x1 - __uint_as_float(h & 0xffff0000u));
              }
            }
            tmem_st8(slot + 8u * q16, hb);
            tmem_st8(slot + kFwdBK / 2 + 8u * q16, lb);
          }
          tmem_wait_st();
          if (kb < f.kb1) n0 += blk;
          tc_fence_before();
          __syncwarp();
          bool yok = true;
          if (lane == 0) {
            mbar_arrive(xempty0 + 8u * xs);   // the raw box is consumed
            // the operand slot is written; its arrival also waits for the
            // stage's N-side tile, so that the MMA lane, whose every
            // shared-memory access costs hundreds of cycles while MMAs are
            // in flight, waits on one barrier per K block
            yok = wait_bounded(yfull0 + 8u * ss, sph, ctl, p.err, 7);
            if (yok) mbar_arrive(tconv0 + 8u * ss);
          }
          if (!__shfl_sync(0xffffffffu, yok ? 1 : 0, 0)) {
            ok = false;
            break;
          }
          if (++xs == SX) {
            xs = 0;
            xph ^= 1u;
          }
          if (++ss == S) {
            ss = 0;
            sph ^= 1u;
          }
        }
        if (!ok) break;
        const int grow = mt * kBM + row;
        // the CTA's last segment: its MMAs and all loads are done, so the
        // operand rings are free to stage this warp's rows of B
        const bool staged = norm && p.stage_b && hi == u_begin;
        // ---- epilogue of this segment
        const bool got = wait_bounded(accf, aphase, ctl, p.err, 5);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (norm) {
          const bool valid = grow < p.M;
          // <B_i, D_i>: lane i reads row i of B with 128-bit loads, two
          // 32-column chunks ahead of the tensor-memory chunk it multiplies
          float dot = 0.0f;
          const int nchk = (f.NC + 31) >> 5;
          const int cbase = nc * f.NC;
          const int ncol = min(f.NC, p.r - cbase);
          const float *brow = p.Bk + static_cast<size_t>(valid ? grow : 0) * p.ldb + cbase;
          if (staged) {
            // 32 x 32 boxes of B (128-byte rows, 128-byte swizzle), one per
            // 32-column chunk, all in flight at once
            const uint32_t region = smem_u32(smem) + static_cast<uint32_t>(quad * nchk) * 4096u;
            const uint32_t sb = stg0 + 8u * quad;
            if (lane == 0) {
              fence_proxy_async_shared();   // the converters' reads of the X ring come first
              mbar_expect_tx(sb, static_cast<uint32_t>(nchk) * 4096u);
              for (int ci = 0; ci < nchk; ++ci)
                tma_load_2d(region + 4096u * ci, &mBs, cbase + 32 * ci, mt * kBM + quad * 32, sb);
            }
            const bool got_b = wait_bounded(sb, 0, ctl, p.err, 11);
            if (!__all_sync(0xffffffffu, got_b)) {
              ok = false;
              break;
            }
            const uint8_t *rw = smem + quad * nchk * 4096 + lane * 128;
            for (int ci = 0; ci < nchk; ++ci) {
              float v[32];
              acc_ld32(32 * ci, v);
              // columns past the chunk's last valid one: neither B (the box may
              // reach into the next chunk) nor the accumulator (past N it was
              // never written) may enter the sum
#pragma unroll
              for (int e = 0; e < 32; ++e)
                if (32 * ci + e >= ncol) v[e] = 0.0f;
              const float4 *bx = reinterpret_cast<const float4 *>(rw + 4096 * ci);
#pragma unroll
              for (int q = 0; q < 8; ++q) {
                float4 bq = bx[q ^ (lane & 7)];
                if (32 * ci + 4 * q >= ncol) bq = make_float4(0.f, 0.f, 0.f, 0.f);
                dot = fmaf(bq.x, v[4 * q], dot);
                dot = fmaf(bq.y, v[4 * q + 1], dot);
                dot = fmaf(bq.z, v[4 * q + 2], dot);
                dot = fmaf(bq.w, v[4 * q + 3], dot);
              }
            }
          } else {
          auto ldb8 = [&](int ci, float4 (&d)[8]) {
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const int c = 32 * ci + 4 * q;
              d[q] = (valid && ci < nchk && c < ncol) ? __ldg(reinterpret_cast<const float4 *>(brow + c))
                                                      : make_float4(0.f, 0.f, 0.f, 0.f);
            }
          };
          float4 b0[8], b1[8], b2[8];
          ldb8(0, b0);
          ldb8(1, b1);
          for (int ci = 0; ci < nchk; ++ci) {
            ldb8(ci + 2, b2);
            float v[32];
            acc_ld32(32 * ci, v);
            // accumulator columns past the chunk's valid ones (past N they
            // were never written) stay out of the sum
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (32 * ci + e >= ncol) v[e] = 0.0f;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              dot = fmaf(b0[q].x, v[4 * q], dot);
              dot = fmaf(b0[q].y, v[4 * q + 1], dot);
              dot = fmaf(b0[q].z, v[4 * q + 2], dot);
              dot = fmaf(b0[q].w, v[4 * q + 3], dot);
            }
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              b0[q] = b1[q];
              b1[q] = b2[q];
            }
          }
          }
          // this segment's records: piece t + cl (see FwdPhase::part)
          float2 *part2 = reinterpret_cast<float2 *>(f.part);
          if (valid) part2[(static_cast<size_t>(t) + cl) * kBM + row] = make_float2(n0, dot);
          // count this warp's 32 records of the M tile; the warp that writes
          // the last ones sums all of them (chunks in order, segments in
          // order) into n_i = sqrt(max(0, sum n0 + 2 s sum dot)), g_i = m_i / n_i
          __threadfence();
          __syncwarp();
          int old = 0;
          if (lane == 0) old = atomicAdd(p.cnt + mt * 4 + quad, 1);
          old = __shfl_sync(0xffffffffu, old, 0);
          int expect = 0;
          for (int c = 0; c < f.nchunks; ++c) {
            const long long ub = (static_cast<long long>(mt) * f.nchunks + c) * f.kbtot;
            expect += split_cta_of(p.ub, f.ctas, ub + f.kbtot - 1) - split_cta_of(p.ub, f.ctas, ub) + 1;
          }
          if (old == expect - 1) {
            __threadfence();
            if (valid) {
              float s0 = 0.0f, sd = 0.0f;
              for (int c = 0; c < f.nchunks; ++c) {
                const long long tc = static_cast<long long>(mt) * f.nchunks + c;
                const int c0 = split_cta_of(p.ub, f.ctas, tc * f.kbtot);
                const int c1 = split_cta_of(p.ub, f.ctas, (tc + 1) * f.kbtot - 1);
                for (int j = c0; j <= c1; ++j) {
                  const float2 v = __ldcg(part2 + (static_cast<size_t>(tc) + j) * kBM + row);
                  if (c == 0) s0 += v.x;
                  sd += v.y;
                }
              }
              const float nn = sqrtf(fmaxf(fmaf(p.two_s, sd, s0), 0.0f));
              p.norm[grow] = nn;
              p.g[grow] = p.m[grow] / nn;
            }
          }
        } else {
          // this CTA's Gram piece (rows of G beyond r are zero: the map of A
          // fills them with zeros)
          float *dst = f.part + (static_cast<size_t>(cl) * kBM + row) * f.NC;
          for (int c = 0; c < f.NC; c += 32) {
            float v[32];
            acc_ld32(c, v);
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
              if (c + j < f.NC) *reinterpret_cast<float4 *>(dst + c + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acce);
        aphase ^= 1u;
      }
      if (ph == 0 && ok && cl < f.P * f.tiles) {
        // ---- this warp's part of the piece is written; once all P pieces of
        // the tile are, reduce this CTA's share of its blocks.  Warps signal
        // and wait on their own (no barrier spans the converter warps), so an
        // abort in one cannot leave another waiting without a bound.
        const int tg = cl / f.P, q = cl - tg * f.P;
        __threadfence();
        __syncwarp();
        if (lane == 0) atomicAdd(p.sync + 1 + tg, 1);
        const bool got = wait_count(p.sync + 1 + tg, 4 * f.P, ctl, p.err, 9);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        __threadfence();
        // blocks of 32 x 32 entries of tile tg: q, q + P, ..., two at a time;
        // thread ct takes 4 consecutive columns (one float4) of two rows of
        // each.  The loads of eight pieces of both blocks are issued before
        // any of them is added; each entry sums the pieces in order.
        int gmt, gnc;
        tile_coords(tg, f.nchunks, 1, &gmt, &gnc);
        const int nsub = (f.NC + 31) / 32;
        const int nmine = (nsub * nsub - q + f.P - 1) / f.P;
        const int c4 = (ct & 7) * 4, r2 = (ct >> 3) * 2;
        const float4 *part4 = reinterpret_cast<const float4 *>(f.part);
        const size_t piece4 = static_cast<size_t>(kBM) * f.NC / 4;
        for (int k0 = 0; k0 < nmine; k0 += 2) {
          int cc[2], rr[2];
          bool vb[2];
#pragma unroll
          for (int kk = 0; kk < 2; ++kk) {
            const int sub = q + (k0 + kk) * f.P;
            const int sr = sub / nsub, sc = sub - sr * nsub;
            vb[kk] = k0 + kk < nmine;
            cc[kk] = sc * 32 + c4;   // first of 4 columns within the tile
            rr[kk] = sr * 32 + r2;   // first of 2 rows within the tile
            vb[kk] = vb[kk] && cc[kk] < f.NC;
          }
          float4 acc[2][2];
#pragma unroll
          for (int kk = 0; kk < 2; ++kk)
#pragma unroll
            for (int e = 0; e < 2; ++e) acc[kk][e] = make_float4(0.f, 0.f, 0.f, 0.f);
          for (int j0 = 0; j0 < f.P; j0 += 8) {
            float4 a[2][8][2];
#pragma unroll
            for (int kk = 0; kk < 2; ++kk)
#pragma unroll
              for (int jj = 0; jj < 8; ++jj)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                  const bool ld = vb[kk] && j0 + jj < f.P && rr[kk] + e < f.NC;
                  const size_t off = (static_cast<size_t>(tg) * f.P + j0 + jj) * piece4 +
                                     (static_cast<size_t>(rr[kk] + e) * f.NC + cc[kk]) / 4;
                  a[kk][jj][e] = ld ? __ldcg(part4 + off) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
            for (int kk = 0; kk < 2; ++kk)
#pragma unroll
              for (int jj = 0; jj < 8; ++jj)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                  acc[kk][e].x += a[kk][jj][e].x;
                  acc[kk][e].y += a[kk][jj][e].y;
                  acc[kk][e].z += a[kk][jj][e].z;
                  acc[kk][e].w += a[kk][jj][e].w;
                }
          }
#pragma unroll
          for (int kk = 0; kk < 2; ++kk) {
            if (!vb[kk]) continue;
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int gr = gmt * f.NC + rr[kk] + e;   // row of G
              if (rr[kk] + e >= f.NC || gr >= p.npad) continue;
              const float w[4] = {acc[kk][e].x, acc[kk][e].y, acc[kk][e].z, acc[kk][e].w};
#pragma unroll
              for (int x = 0; x < 4; ++x) {
                const int gc = gnc * f.NC + cc[kk] + x;   // column of G
                if (gc >= p.npad) continue;
                const float v = (gr < p.r && gc < p.r) ? p.half_s * w[x] : 0.0f;
                store_gs3(p.gs_h, p.gs_l, p.npad, gr, gc, v);
                if (gmt != gnc) store_gs3(p.gs_h, p.gs_l, p.npad, gc, gr, v);
              }
            }
          }
        }
        // s/2 G is read by the other CTAs' TMA loads (async proxy)
        __threadfence();
        fence_proxy_async_global();
        __syncwarp();
        if (lane == 0) atomicAdd(p.sync + 0, 1);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem, static_cast<uint32_t>(p.tmem_cols));
  }
}

// ---------------------------------------------------------------------------
// elementwise helpers
// ---------------------------------------------------------------------------

// N-side split of a [rows, cols] fp32 matrix for the bf16 three-product
// scheme, and zero fill of the norm pass's ncnt completion counters:
//   h [rows, cols8] bf16: x rounded to bf16 (nearest even)
//   l [rows, cols8] bf16: x - h rounded to bf16;  zero past cols
// (cols8 = cols rounded up to 8, a 16-byte row).  One thread per group of 4.
__device__ __forceinline__ void split_hl_range(const float *__restrict__ x, long long rows, int cols, int cols8,
                                               __nv_bfloat16 *__restrict__ h, __nv_bfloat16 *__restrict__ l,
                                               long long first, long long step) {
  const int g4 = cols8 / 4;
  const long long n = rows * g4;
  for (long long i = first; i < n; i += step) {
    const long long row = i / g4;
    const int k = static_cast<int>(i - row * g4) * 4;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (k < cols) v = __ldg(reinterpret_cast<const float4 *>(x + row * cols + k));
    const uint32_t h01 = pack_bf16x2(v.x, v.y), h23 = pack_bf16x2(v.z, v.w);
    const uint32_t l01 = pack_bf16x2(v.x - __uint_as_float(h01 << 16), v.y - __uint_as_float(h01 & 0xffff0000u));
    const uint32_t l23 = pack_bf16x2(v.z - __uint_as_float(h23 << 16), v.w - __uint_as_float(h23 & 0xffff0000u));
    *reinterpret_cast<uint2 *>(h + row * cols8 + k) = make_uint2(h01, h23);
    *reinterpret_cast<uint2 *>(l + row * cols8 + k) = make_uint2(l01, l23);
  }
}

__global__ void __launch_bounds__(256) split_hl_kernel(const float *__restrict__ x, long long rows, int cols,
                                                       int cols8, __nv_bfloat16 *__restrict__ h,
                                                       __nv_bfloat16 *__restrict__ l, int *__restrict__ cnt,
                                                       int ncnt) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < ncnt; i += gridDim.x * blockDim.x) cnt[i] = 0;
  split_hl_range(x, rows, cols, cols8, h, l, static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x,
                 static_cast<long long>(gridDim.x) * blockDim.x);
}

// B [out, r] -> Bp [out, rp] with zero columns r..rp-1 (rp = r rounded up to 4)
__global__ void __launch_bounds__(256) pad_cols_kernel(const float *__restrict__ B, long long rows, int r, int rp,
                                                       float *__restrict__ Bp) {
  const long long n = rows * rp;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const long long row = i / rp;
    const int c = static_cast<int>(i - row * rp);
    Bp[i] = c < r ? B[row * r + c] : 0.0f;
  }
}

// how partial results were laid out by tc_gemm_kernel: tile t = (M tile, N
// chunk) is covered by CTAs cta_of(t*kbtot) .. cta_of((t+1)*kbtot - 1); the
// partial of M tile mt, chunk nc, from the j-th of those CTAs, is entry
// (mt*nchunks + nc)*maxseg + j
struct StreamK {
  long long units;
  int ncl, kbtot, maxseg;
};

// entry (a, b) of a Gram result v, zero-padded to [npad, npad] and split for
// the N side: h [npad, npad] = bf16(v), l [npad, npad] = bf16(v - h)
__device__ __forceinline__ void store_gs_hl(int a, int b, float v, int npad, __nv_bfloat16 *gh, __nv_bfloat16 *gl) {
  if (a >= npad || b >= npad) return;
  const __nv_bfloat16 h = __float2bfloat16_rn(v);
  const long long i = static_cast<long long>(a) * npad + b;
  gh[i] = h;
  gl[i] = __float2bfloat16_rn(v - __bfloat162float(h));
}

// One 32 x 32 block of an upper-triangular Gram tile (blockIdx.x = tile, whose
// M tile is mt and N chunk nc >= mt; blockIdx.y = block in the tile).  Warp w
// sums the segments w, w + 8, ... of the tile's partials (a lane per column,
// 32 independent row sums, so the loads of a segment are in flight together);
// the 8 warp sums are then added in warp order.  The block is written at
// (k, l) and, for a tile off the diagonal, mirrored at (l, k) through shared
// memory, so both writes are coalesced.
// The result is written split, as the bf16 h and l [npad, npad] (store_gs_hl).
__global__ void __launch_bounds__(256) gram_reduce_kernel(const float *__restrict__ part, StreamK sk, int nchunks,
                                                          int NC, int r, int npad, float half_s,
                                                          __nv_bfloat16 *__restrict__ gh, __nv_bfloat16 *__restrict__ gl) {
  auto store = [&](int a, int b, float v) { store_gs_hl(a, b, v, npad, gh, gl); };
  __shared__ float wsum[8][32][33];
  const int t = blockIdx.x;
  int mt, nc;
  tile_coords(t, nchunks, 1, &mt, &nc);
  const int nsub = (NC + 31) / 32;
  const int sr = static_cast<int>(blockIdx.y) / nsub, sc = static_cast<int>(blockIdx.y) - sr * nsub;
  const size_t tm = static_cast<size_t>(mt) * nchunks + nc;
  const long long ub = static_cast<long long>(t) * sk.kbtot;
  const int nseg = cta_of(ub + sk.kbtot - 1, sk.units, sk.ncl) - cta_of(ub, sk.units, sk.ncl) + 1;
  const int tx = threadIdx.x, ty = threadIdx.y;
  // valid rows of this block (G has r rows and columns) and this lane's column
  const int nrow = min(32, min(kBM, r - mt * kBM) - sr * 32);
  const int col = sc * 32 + tx;
  const bool cvalid = col < NC && nc * NC + col < r;
  float acc[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) acc[i] = 0.0f;
  if (cvalid) {
    for (int j = ty; j < nseg; j += 8) {
      const float *pj = part + ((tm * sk.maxseg + j) * kBM + sr * 32) * NC + col;
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (i < nrow) acc[i] += pj[static_cast<size_t>(i) * NC];
    }
  }
#pragma unroll
  for (int i = 0; i < 32; ++i) wsum[ty][i][tx] = acc[i];
  __syncthreads();
  float v[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int i = ty + 8 * q;
    float sum = 0.0f;
#pragma unroll
    for (int w = 0; w < 8; ++w) sum += wsum[w][i][tx];
    v[q] = (i < nrow && cvalid) ? half_s * sum : 0.0f;
  }
  __syncthreads();
  // wsum[0] now holds the block's values for the mirrored write
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int i = ty + 8 * q;
    store(mt * kBM + sr * 32 + i, nc * NC + col, v[q]);
    wsum[0][i][tx] = v[q];
  }
  if (mt != nc) {
    __syncthreads();
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int i = ty + 8 * q;
      store(nc * NC + sc * 32 + i, mt * kBM + sr * 32 + tx, wsum[0][tx][i]);
    }
  }
}

// ---------------------------------------------------------------------------
// gradient through the norm (norm not detached)
//
// With c_i = (dL/dn_i) / n_i and dL/dn_i = -g_i d_mag_i (d_mag = dL/dm along
// g = m / n), and V = W0 + s B A:
//     dB   = s c (.) (W0 A^T + s B G)                 G = A A^T
//     dA^T = W0^T (s c (.) B) + A^T (s^2 H)           H = B^T diag(c) B
// Both are the norm pass's GEMM shape: dB is [W0 | B] x [A | sG]^T over
// K = in + r with rows scaled by s c_i at the end; dA^T is [W0^T | A^T] x
// [(s c B)^T | s^2 H]^T over K = out + r, its M-side operands read transposed.
// ---------------------------------------------------------------------------

// Y = (s c (.) B)^T [r, out8], columns out..out8-1 zero, split for the N side
// like split_hl_kernel: h and l [r, out8] bf16.  One block (bx, by) of 256
// threads transposes 32 rows of B by 128 of its columns (four 32 x 32 tiles
// through shared memory, all sixteen loads of a thread in flight together);
// the rows' coefficients s c_i are formed once per block.
constexpr int kBsCols = 128;   // columns of B (rows of Y) per block
__device__ __forceinline__ void bs_split_block(long long bx, int by, const float *__restrict__ B, long long out,
                                               int r, long long out8, const float *__restrict__ g,
                                               const float *__restrict__ d_mag, const float *__restrict__ norm,
                                               float s, __nv_bfloat16 *__restrict__ yh,
                                               __nv_bfloat16 *__restrict__ yl, float *smem) {
  float(*tile)[32][33] = reinterpret_cast<float(*)[32][33]>(smem);   // [kBsCols / 32][32][33]
  float *coef = smem + (kBsCols / 32) * 32 * 33;                      // [32]
  const long long i0 = bx * 32;
  const int n0 = by * kBsCols;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  if (ty == 0) {
    const long long i = i0 + tx;
    coef[tx] = i < out ? s * norm_grad_coef(g, d_mag, norm, i) : 0.0f;
  }
  __syncthreads();
#pragma unroll
  for (int c = 0; c < kBsCols / 32; ++c) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int il = ty + 8 * q;
      const long long i = i0 + il;
      const int n = n0 + 32 * c + tx;
      float v = 0.0f;
      if (i < out && n < r) v = coef[il] * B[i * r + n];
      tile[c][il][tx] = v;
    }
  }
  __syncthreads();
#pragma unroll
  for (int c = 0; c < kBsCols / 32; ++c) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int n = n0 + 32 * c + ty + 8 * q;
      const long long i = i0 + tx;
      if (n < r && i < out8) {
        const float x = tile[c][tx][ty + 8 * q];
        const long long o = static_cast<long long>(n) * out8 + i;
        const __nv_bfloat16 h = __float2bfloat16_rn(x);
        yh[o] = h;
        yl[o] = __float2bfloat16_rn(x - __bfloat162float(h));
      }
    }
  }
}

// ---- the Gram products on the CUDA cores (r <= kSgMaxR)
//
// At small r, G = A A^T (K = in) and s H = B^T (s c (.) B) (K = out) are a few
// hundred MFLOP; as tensor-core passes of their own they are bound by the
// latency of one CTA's K loop and by four launches.  Here a block of the
// gradient's first launch forms one fp32 partial of a T x T tile of the upper
// triangle over one K slice, and the next launch sums the slices of each entry
// in a fixed order.  T (16, 32 or 64, the smallest that covers r up to 64) keeps
// the FMAs on entries below r.  In a block, each thread holds a 4 x 4 block of
// the tile; the (T/4)^2 threads that cover the tile form a K group, and the
// 256 / (T/4)^2 groups take equal parts of each chunk of KC K indices staged
// K-major in shared memory (the next chunk's loads in flight during the FMAs).
// The groups' tiles are added in group order at the end.
constexpr int kSgMaxSlices = 128;   // K slices per tile at most (bounds the partials)
constexpr int kSgMaxR = 256;        // largest r that takes this path
constexpr int kSgSmemFloats = 4672; // staging (and group sums) of a block, floats

template <int T>
struct SgShape {
  static constexpr int kTT = T / 4;                      // threads per tile side
  static constexpr int kGroup = kTT * kTT;               // threads per K group
  static constexpr int kGroups = 256 / kGroup;           // K groups per block
  static constexpr int kKC = T == 64 ? 32 : 64;          // K indices per chunk
  static constexpr int kLd = T + 4;                      // row stride of a K-major chunk (16-byte rows)
  static constexpr int kKK = kKC / kGroups;              // K indices of a chunk per group
  static constexpr int kSlice = T == 16 ? 64 : 128;      // K indices per slice (at most kSgMaxSlices)
  static_assert(kGroups * kGroup == 256 && kKK * kGroups == kKC, "K groups");
  static_assert(2 * kKC * kLd + kKC <= kSgSmemFloats && kGroups * T * T <= kSgSmemFloats, "shared memory");
};

struct SgDims {
  int T;            // tile side (16, 32 or 64); 0: no Gram part
  int nt1;          // tiles per side, ceil(r / T)
  int ntiles;       // upper-triangular tiles, nt1 (nt1 + 1) / 2
  int nsG, nsH;     // K slices of G (K = in) and of H (K = out)
  int ksG, ksH;     // K indices per slice (multiples of the chunk)
};

__host__ __device__ __forceinline__ void sg_tile(int t, int nt1, int *ti, int *tj) {
  int i = 0;
  while (t >= nt1 - i) {
    t -= nt1 - i;
    ++i;
  }
  *ti = i;
  *tj = i + t;
}

// Partial q of the Gram part: q < ntiles * nsG is G's (tile q / nsG, slice
// q % nsG), the rest are H's.  part[q] is the T x T tile, row-major, entries
// past r zero.  A is [r, in] with 16-byte rows (in % 4 == 0), B is [out, r].
template <int T>
__device__ __forceinline__ void sg_part_block(int q, const SgDims &d, const float *__restrict__ A, int r,
                                              long long in, const float *__restrict__ B, long long out,
                                              const float *__restrict__ g, const float *__restrict__ d_mag,
                                              const float *__restrict__ norm, float s, float *__restrict__ part,
                                              float *smem) {
  using S = SgShape<T>;
  constexpr int KC = S::kKC, LD = S::kLd;
  constexpr int NQ = T * KC / 4 / 256;   // float4s of an A chunk per thread and operand (G)
  constexpr int NE = T * KC / 256;       // entries of a B chunk per thread and operand (H)
  const bool isG = q < d.ntiles * d.nsG;
  const int qq = isG ? q : q - d.ntiles * d.nsG;
  const int ns = isG ? d.nsG : d.nsH;
  const int t = qq / ns, z = qq - t * ns;
  int ti, tj;
  sg_tile(t, d.nt1, &ti, &tj);
  const int i0 = ti * T, j0 = tj * T;
  const long long K = isG ? in : out;
  const long long k0 = static_cast<long long>(z) * (isG ? d.ksG : d.ksH);
  const long long kend = min(K, k0 + (isG ? d.ksG : d.ksH));
  const int nch = static_cast<int>((kend - k0 + KC - 1) / KC);
  float(*xi)[LD] = reinterpret_cast<float(*)[LD]>(smem);
  float(*xj)[LD] = (isG && ti == tj) ? xi : reinterpret_cast<float(*)[LD]>(smem + KC * LD);
  float *coef = smem + 2 * KC * LD;   // s c_k of the chunk's rows of B (H)
  const int tid = threadIdx.x;
  const int grp = tid / S::kGroup, loc = tid - grp * S::kGroup;
  const int ty = loc / S::kTT, tx = loc - ty * S::kTT;
  // a chunk's loads, held in registers until staged:
  //   G: NQ quads of A rows per operand, KC / 4 lanes along a row piece
  //   H: NE entries of B per operand, T lanes along a row of B; the first KC
  //      threads also fetch the inputs of one row's coefficient
  float vi[4 * NQ > NE ? 4 * NQ : NE], vj[4 * NQ > NE ? 4 * NQ : NE];
  float cg = 0.0f, cd = 0.0f, cn = 1.0f;
  auto load = [&](long long kc) {
    if (isG) {
#pragma unroll
      for (int e = 0; e < NQ; ++e) {
        const int f = tid + 256 * e;
        const int row = f / (KC / 4), kq = (f - row * (KC / 4)) * 4;
        const long long k = kc + kq;
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
        if (k < kend) {
          if (i0 + row < r) a = __ldg(reinterpret_cast<const float4 *>(A + (i0 + row) * in + k));
          if (ti != tj && j0 + row < r) b = __ldg(reinterpret_cast<const float4 *>(A + (j0 + row) * in + k));
        }
        vi[4 * e] = a.x, vi[4 * e + 1] = a.y, vi[4 * e + 2] = a.z, vi[4 * e + 3] = a.w;
        vj[4 * e] = b.x, vj[4 * e + 1] = b.y, vj[4 * e + 2] = b.z, vj[4 * e + 3] = b.w;
      }
    } else {
#pragma unroll
      for (int e = 0; e < NE; ++e) {
        const int f = tid + 256 * e;
        const int kk = f / T, col = f - kk * T;
        const long long k = kc + kk;
        float a = 0.0f, b = 0.0f;
        if (k < kend) {
          if (i0 + col < r) a = B[k * r + i0 + col];
          if (j0 + col < r) b = B[k * r + j0 + col];
        }
        vi[e] = a;
        vj[e] = b;
      }
      if (tid < KC && kc + tid < kend) {
        cg = g[kc + tid];
        cd = d_mag[kc + tid];
        cn = norm[kc + tid];
      }
    }
  };
  auto stage = [&]() {
    if (isG) {
#pragma unroll
      for (int e = 0; e < NQ; ++e) {
        const int f = tid + 256 * e;
        const int row = f / (KC / 4), kq = (f - row * (KC / 4)) * 4;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          xi[kq + m][row] = vi[4 * e + m];
          if (ti != tj) xj[kq + m][row] = vj[4 * e + m];
        }
      }
    } else {
      // the coefficients first (rows past K get 0: their B entries are 0)
      if (tid < KC) coef[tid] = s * (-(cg * cd) / cn);
      __syncthreads();
#pragma unroll
      for (int e = 0; e < NE; ++e) {
        const int f = tid + 256 * e;
        const int kk = f / T, col = f - kk * T;
        xi[kk][col] = vi[e];
        xj[kk][col] = coef[kk] * vj[e];
      }
    }
  };
  float acc[4][4];
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int b = 0; b < 4; ++b) acc[a][b] = 0.0f;
  load(k0);
  for (int c = 0; c < nch; ++c) {
    __syncthreads();
    stage();
    __syncthreads();
    if (c + 1 < nch) {
      cg = 0.0f, cd = 0.0f, cn = 1.0f;
      load(k0 + static_cast<long long>(c + 1) * KC);
    }
#pragma unroll 8
    for (int u0 = 0; u0 < S::kKK; ++u0) {
      const int kk = grp * S::kKK + u0;
      const float4 a = *reinterpret_cast<const float4 *>(&xi[kk][4 * ty]);
      const float4 b = *reinterpret_cast<const float4 *>(&xj[kk][4 * tx]);
      const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int v = 0; v < 4; ++v) acc[u][v] = fmaf(av[u], bv[v], acc[u][v]);
    }
  }
  float *pp = part + static_cast<size_t>(q) * T * T;
  if constexpr (S::kGroups == 1) {
#pragma unroll
    for (int u = 0; u < 4; ++u)
      *reinterpret_cast<float4 *>(pp + (4 * ty + u) * T + 4 * tx) =
          make_float4(acc[u][0], acc[u][1], acc[u][2], acc[u][3]);
    return;
  }
  // the groups' tiles side by side in shared memory, then added in group order
  __syncthreads();
  float *gs = smem + grp * T * T;
#pragma unroll
  for (int u = 0; u < 4; ++u)
    *reinterpret_cast<float4 *>(gs + (4 * ty + u) * T + 4 * tx) =
        make_float4(acc[u][0], acc[u][1], acc[u][2], acc[u][3]);
  __syncthreads();
  for (int e = tid; e < T * T; e += 256) {
    float v = smem[e];
#pragma unroll
    for (int k = 1; k < S::kGroups; ++k) v += smem[k * T * T + e];
    pp[e] = v;
  }
}

// The gradient's first launch: blocks [0, nb_sg) are Gram partials (T > 0
// only), the next nb_bs the split of (s c (.) B)^T (bs_bx per row of blocks),
// the last nb_split the split of A (split_hl_kernel's work, grid stride).
// The three parts read only the call's inputs, so they run side by side; the
// Gram blocks, the longest, come first.
struct GradPrep {
  SgDims sg;
  int nb_sg, nb_bs, bs_bx, nb_split;
  const float *A;
  int r, in, in8;
  __nv_bfloat16 *a_h, *a_l;
  const float *B;
  long long out, out8;
  const float *g, *d_mag, *norm;
  float s;
  __nv_bfloat16 *y_h, *y_l;
  float *sg_part;
};
static_assert(kSgSmemFloats >= (kBsCols / 32) * 32 * 33 + 32, "prep shared memory holds the bs_split tiles");

template <int T>
__global__ void __launch_bounds__(256, 3) grad_prep_kernel(const GradPrep p) {
  __shared__ __align__(16) float smem[T > 0 ? kSgSmemFloats : (kBsCols / 32) * 32 * 33 + 32];
  int b = static_cast<int>(blockIdx.x);
  if constexpr (T > 0) {
    if (b < p.nb_sg) {
      sg_part_block<T>(b, p.sg, p.A, p.r, p.in, p.B, p.out, p.g, p.d_mag, p.norm, p.s, p.sg_part, smem);
      return;
    }
    b -= p.nb_sg;
  }
  if (b < p.nb_bs) {
    bs_split_block(b % p.bs_bx, b / p.bs_bx, p.B, p.out, p.r, p.out8, p.g, p.d_mag, p.norm, p.s, p.y_h, p.y_l, smem);
    return;
  }
  b -= p.nb_bs;
  split_hl_range(p.A, p.r, p.in, p.in8, p.a_h, p.a_l, static_cast<long long>(b) * blockDim.x + threadIdx.x,
                 static_cast<long long>(p.nb_split) * blockDim.x);
}

// Sum of the Gram partials: warp w adds slices w, w + 8, ... in turn, then the
// 8 warp sums are added in warp order; times s (s G from G, s^2 H from s H),
// written split into the bf16 h / l [npad, npad] the passes read, mirrored
// below the diagonal (zero past r, as the partials are).  blockIdx.x =
// (product * ntiles + tile) * (T^2 / 64) + entry group; a block covers 64
// consecutive entries of a tile (row-major), two per lane.
__global__ void __launch_bounds__(256) sg_fin_kernel(const float *__restrict__ part, const SgDims d, int npad,
                                                     float s, __nv_bfloat16 *__restrict__ gh,
                                                     __nv_bfloat16 *__restrict__ gl, __nv_bfloat16 *__restrict__ hh,
                                                     __nv_bfloat16 *__restrict__ hl) {
  __shared__ float wsum[8][2][33];
  const int T = d.T, tt = T * T, per = tt / 64;
  int b = static_cast<int>(blockIdx.x);
  const int eg = b % per;
  b /= per;
  const bool isG = b < d.ntiles;
  const int t = isG ? b : b - d.ntiles;
  const int ns = isG ? d.nsG : d.nsH;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const float *p0 = part + ((isG ? 0 : static_cast<size_t>(d.ntiles) * d.nsG) + static_cast<size_t>(t) * ns) * tt +
                    eg * 64 + lane;
  float acc[2] = {0.0f, 0.0f};
#pragma unroll 8
  for (int z = w; z < ns; z += 8) {
    const float *pz = p0 + static_cast<size_t>(z) * tt;
    acc[0] += __ldcg(pz);
    acc[1] += __ldcg(pz + 32);
  }
  wsum[w][0][lane] = acc[0];
  wsum[w][1][lane] = acc[1];
  __syncthreads();
  if (threadIdx.x < 64) {
    const int a = threadIdx.x >> 5;
    float v = 0.0f;
#pragma unroll
    for (int k = 0; k < 8; ++k) v += wsum[k][a][lane];
    v *= s;
    int ti, tj;
    sg_tile(t, d.nt1, &ti, &tj);
    const int e = eg * 64 + a * 32 + lane;
    const int row = ti * T + e / T, col = tj * T + e % T;
    __nv_bfloat16 *oh = isG ? gh : hh, *ol = isG ? gl : hl;
    store_gs_hl(row, col, v, npad, oh, ol);
    if (ti != tj) store_gs_hl(col, row, v, npad, oh, ol);
  }
}

// Sum of the parts of a ROWS pass, in part order.  blockIdx.x = M tile *
// nchunks + N chunk, blockIdx.y = block of 32 columns of the chunk; warp w
// takes column group 8 * blockIdx.y + w (4 columns, float4 partials) for the
// tile's 128 rows, lanes along rows.
//   trans = 0: out[row][col] = s c_row * sum, through shared memory so that a
//              warp writes 32 consecutive columns of a row          (dB)
//   trans = 1: out[col][row] = sum, lanes along rows                (dA)
__global__ void __launch_bounds__(256) rows_reduce_kernel(const float4 *__restrict__ part, StreamK sk, int nchunks,
                                                          int NC, int M, int ncols, int trans,
                                                          const float *__restrict__ g,
                                                          const float *__restrict__ d_mag,
                                                          const float *__restrict__ norm, float s,
                                                          float *__restrict__ out, long long ldo) {
  __shared__ float tile[kBM][33];
  __shared__ float coef[kBM];   // s c_row of the block's rows (dB)
  const int tm = blockIdx.x;
  const int mt = tm / nchunks, nc = tm - mt * nchunks;
  const long long ub = (static_cast<long long>(mt) * nchunks + nc) * sk.kbtot;
  const int nseg = cta_of(ub + sk.kbtot - 1, sk.units, sk.ncl) - cta_of(ub, sk.units, sk.ncl) + 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cg = static_cast<int>(blockIdx.y) * 8 + warp;   // column group within the chunk
  const int ncol = min(NC, ncols - nc * NC);                 // valid columns of the chunk
  const size_t slot = static_cast<size_t>(32) * NC;          // float4s per part
  const long long row0 = static_cast<long long>(mt) * kBM;
  const float4 *src = part + static_cast<size_t>(tm) * sk.maxseg * slot + static_cast<size_t>(cg) * kBM + lane;
  float4 acc[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (!trans && threadIdx.x < kBM) {
    const long long row = row0 + threadIdx.x;
    coef[threadIdx.x] = row < M ? s * norm_grad_coef(g, d_mag, norm, row) : 0.0f;
  }
  if (4 * cg < ncol) {
    // parts in order, two parts' loads in flight per round
    auto part4 = [&](int j, float4 (&o)[4]) {
#pragma unroll
      for (int k = 0; k < 4; ++k)
        o[k] = (j < nseg && row0 + 32 * k + lane < M) ? __ldcg(src + j * slot + 32 * k)
                                                      : make_float4(0.f, 0.f, 0.f, 0.f);
    };
    auto add4 = [&](const float4 (&o)[4]) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        acc[k].x += o[k].x;
        acc[k].y += o[k].y;
        acc[k].z += o[k].z;
        acc[k].w += o[k].w;
      }
    };
    for (int j = 0; j < nseg; j += 2) {
      float4 o0[4], o1[4];
      part4(j, o0);
      part4(j + 1, o1);
      add4(o0);
      if (j + 1 < nseg) add4(o1);
    }
  }
  if (trans) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const long long row = row0 + 32 * k + lane;
      const float w[4] = {acc[k].x, acc[k].y, acc[k].z, acc[k].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int col = 4 * cg + e;
        if (row < M && col < ncol) out[(static_cast<long long>(nc) * NC + col) * ldo + row] = w[e];
      }
    }
    return;
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    tile[32 * k + lane][4 * warp + 0] = acc[k].x;
    tile[32 * k + lane][4 * warp + 1] = acc[k].y;
    tile[32 * k + lane][4 * warp + 2] = acc[k].z;
    tile[32 * k + lane][4 * warp + 3] = acc[k].w;
  }
  __syncthreads();
  const int col = static_cast<int>(blockIdx.y) * 32 + lane;
  for (int rr = warp; rr < kBM; rr += 8) {
    const long long row = row0 + rr;
    if (row < M && col < ncol)
      out[row * ldo + static_cast<long long>(nc) * NC + col] = coef[rr] * tile[rr][lane];
  }
}

// ---------------------------------------------------------------------------
// bf16 weights: W0, A, B in bf16 make every product exact in fp32, so the
// contraction is one kind::f16 MMA per 16 K indices with both operands taken
// from shared memory as TMA delivers them (no split, no converter warps).  The
// Gram part of the fold needs s/2 G at fp32 precision: it is split into three
// bf16 pieces h1 + h2 + h3 (each the bf16 rounding of what is left) laid side by
// side along K, against B repeated three times.  ||W0_i||^2 is an input (W0 is
// frozen during fine-tuning, so its row norms are computed once).
// ---------------------------------------------------------------------------
struct Tc16Params {
  int mode;
  int M;            // valid M-side rows (out, or r for the Gram pass)
  int kb1;          // K blocks over in (W0 or A columns)
  int kbr;          // K blocks over r (one piece of the Gram part)
  int rs;           // column stride of the pieces of s/2 G (r rounded up to 8)
  int kbtot;        // kb1 + 3 * kbr (NORM) or kb1 (GRAM)
  int nchunks, sym, NC;
  int nbox, nb, NT;
  int nmma0, nmma1;
  int tmem_cols;
  int stages;
  int tiles;
  long long units;
  int ctas, ncl, maxseg;
  unsigned stage_bytes, x_bytes;
  float *part;
  int r;
  int *err;
  int *cnt;
  const float *m;
  const float *n0sq;                 // ||W0_i||^2, fp32 [M]
  float *norm, *g;
  float two_s;
  const __nv_bfloat16 *Bk;           // B [M, ldb] bf16 (the epilogue reads its rows)
  int ldb;
};

// BKE bf16 per K block: 32 (64-byte rows, 64-byte swizzle) or 64 (128-byte rows,
// 128-byte swizzle); the matching descriptor is sdesc<BKE / 2>.
template <int BKE>
__global__ void __launch_bounds__(kThreads, 1)
tc16_kernel(const __grid_constant__ CUtensorMap mX1, const __grid_constant__ CUtensorMap mX2,
            const __grid_constant__ CUtensorMap mY1, const __grid_constant__ CUtensorMap mY2, const Tc16Params p) {
  constexpr int kRowBytes = BKE * 2;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int S = p.stages;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + static_cast<size_t>(S) * p.stage_bytes);
  // barrier layout: full[S], empty[S], accf, acce, fin
  SharedCtl *ctl = reinterpret_cast<SharedCtl *>(bars + 2 * S + 3);
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = full0 + 8u * S;
  const uint32_t accf = empty0 + 8u * S;
  const uint32_t acce = accf + 8;
  const uint32_t fin = acce + 8;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full0 + 8u * s, 1);
      mbar_init(empty0 + 8u * s, 1);
    }
    mbar_init(accf, 1);
    mbar_init(acce, 4);
    mbar_init(fin, 1);
    ctl->abort = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_map(&mX1);
    prefetch_map(&mY1);
    if (p.kbtot > p.kb1) {
      prefetch_map(&mX2);
      prefetch_map(&mY2);
    }
  }
  if (warp == 1) {
    __syncwarp();
    tmem_alloc(smem_u32(&ctl->tmem_base), static_cast<uint32_t>(p.tmem_cols));
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  const int cl = static_cast<int>(blockIdx.x);
  const long long u_begin = unit_begin(cl, p.units, p.ncl);
  const long long u_end = unit_begin(cl + 1, p.units, p.ncl);

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      bool ok = *reinterpret_cast<volatile int *>(&g_dora_stall) == 0;
      for (long long u = u_begin; u < u_end && ok;) {
        const int t = static_cast<int>(u / p.kbtot);
        const int kb0 = static_cast<int>(u - static_cast<long long>(t) * p.kbtot);
        const int kbe = static_cast<int>(min(static_cast<long long>(p.kbtot), kb0 + (u_end - u)));
        int mt, nc;
        tile_coords(t, p.nchunks, p.sym, &mt, &nc);
        for (int kb = kb0; kb < kbe; ++kb) {
          if (!wait_bounded(empty0 + 8u * stage, phase ^ 1u, ctl, p.err, 1)) {
            ok = false;
            break;
          }
          const uint32_t fb = full0 + 8u * stage;
          mbar_expect_tx(fb, p.stage_bytes);
          const uint32_t xs = smem_u32(smem + static_cast<size_t>(stage) * p.stage_bytes);
          const uint32_t ys = xs + p.x_bytes;
          if (kb < p.kb1) {
            const int kx = kb * BKE;
            tma_load_2d(xs, &mX1, kx, mt * kBM, fb);
            for (int i = 0; i < p.nb; ++i)
              tma_load_2d(ys + static_cast<uint32_t>(i * p.nbox * kRowBytes), &mY1, kx, nc * p.NC + i * p.nbox, fb);
          } else {
            // Gram part: K block kb2 of B (repeated for each piece) against piece kb2 / kbr of s/2 G
            const int kb2 = kb - p.kb1;
            const int piece = kb2 / p.kbr, kc = (kb2 - piece * p.kbr) * BKE;
            tma_load_2d(xs, &mX2, kc, mt * kBM, fb);
            for (int i = 0; i < p.nb; ++i)
              tma_load_2d(ys + static_cast<uint32_t>(i * p.nbox * kRowBytes), &mY2, piece * p.rs + kc,
                          nc * p.NC + i * p.nbox, fb);
          }
          ++issued;
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        u += kbe - kb0;
      }
      if (!ok) {
        int st = stage;
        uint32_t ph = phase;
        for (int k = 0; k < S && k < issued; ++k) {
          if (--st < 0) {
            st = S - 1;
            ph ^= 1u;
          }
          wait_drain(full0 + 8u * st, ph);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      int stage = 0;
      uint32_t phase = 0;
      uint32_t aphase = 0;
      bool ok = true;
      const uint32_t ic0 = idesc_bf16(p.nmma0);
      const uint32_t ic1 = p.nmma1 > 0 ? idesc_bf16(p.nmma1) : 0u;
      for (long long u = u_begin; u < u_end && ok;) {
        const int t = static_cast<int>(u / p.kbtot);
        const int kb0 = static_cast<int>(u - static_cast<long long>(t) * p.kbtot);
        const int kbe = static_cast<int>(min(static_cast<long long>(p.kbtot), kb0 + (u_end - u)));
        if (!wait_bounded(acce, aphase ^ 1u, ctl, p.err, 3)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int kb = kb0; kb < kbe; ++kb) {
          if (!wait_bounded(full0 + 8u * stage, phase, ctl, p.err, 2)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t xs = smem_u32(smem + static_cast<size_t>(stage) * p.stage_bytes);
          const uint32_t ys = xs + p.x_bytes;
#pragma unroll
          for (int k = 0; k < BKE / 16; ++k) {
            const uint32_t acc0 = (kb != kb0 || k != 0) ? 1u : 0u;
            const uint32_t ko = static_cast<uint32_t>(k) * 32u;   // 16 bf16
            const uint64_t a = sdesc<BKE / 2>(xs + ko);
            mma_bf16_ss(tmem, a, sdesc<BKE / 2>(ys + ko), ic0, acc0);
            if (p.nmma1 > 0) mma_bf16_ss(tmem + 256u, a, sdesc<BKE / 2>(ys + 256u * kRowBytes + ko), ic1, acc0);
          }
          mma_commit(empty0 + 8u * stage);
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(accf);
        aphase ^= 1u;
        u += kbe - kb0;
      }
      mma_commit(fin);
      wait_drain(fin, 0);
    }
  } else if (warp >= 2 && warp <= 5) {
    // ---------------------------------------------------------------- epilogue
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    uint32_t aphase = 0;
    bool ok = true;
    for (long long u = u_begin; u < u_end && ok;) {
      const int t = static_cast<int>(u / p.kbtot);
      const int kb0 = static_cast<int>(u - static_cast<long long>(t) * p.kbtot);
      const int kbe = static_cast<int>(min(static_cast<long long>(p.kbtot), kb0 + (u_end - u)));
      int mt, nc;
      tile_coords(t, p.nchunks, p.sym, &mt, &nc);
      const size_t tm = static_cast<size_t>(mt) * p.nchunks + nc;
      if (p.mode == kNorm && lane == 0) {
        const int r0 = mt * kBM + quad * 32;
        const int nr = min(32, p.M - r0);
        if (nr > 0)
          prefetch_l2(p.Bk + static_cast<size_t>(r0) * p.ldb, static_cast<uint32_t>(nr) * p.ldb * 2u);
      }
      const int grow = mt * kBM + row;
      const bool valid = grow < p.M;
      const int seg = cl - cta_of(static_cast<long long>(t) * p.kbtot, p.units, p.ncl);
      const bool got = wait_bounded(accf, aphase, ctl, p.err, 5);
      if (!__all_sync(0xffffffffu, got)) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (p.mode == kNorm) {
        // <B_i, D_i>: lane i reads row i of B (bf16, 8 per 128-bit load)
        float dot = 0.0f;
        const int nchk = (p.NC + 31) >> 5;
        const int cbase = nc * p.NC;
        const int ncol = min(p.NC, p.r - cbase);
        const __nv_bfloat16 *brow = p.Bk + static_cast<size_t>(valid ? grow : 0) * p.ldb + cbase;
        for (int ci = 0; ci < nchk; ++ci) {
          uint4 bq[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int c = 32 * ci + 8 * q;
            bq[q] = (valid && c < ncol) ? __ldg(reinterpret_cast<const uint4 *>(brow + c)) : make_uint4(0, 0, 0, 0);
          }
          float v[32];
          tmem_ld32(lane_addr + static_cast<uint32_t>(32 * ci), v);
          // accumulator columns past the chunk's valid ones (past N they were
          // never written) stay out of the sum
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (32 * ci + e >= ncol) v[e] = 0.0f;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint32_t w[4] = {bq[q].x, bq[q].y, bq[q].z, bq[q].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              dot = fmaf(__uint_as_float(w[e] << 16), v[8 * q + 2 * e], dot);
              dot = fmaf(__uint_as_float(w[e] & 0xffff0000u), v[8 * q + 2 * e + 1], dot);
            }
          }
        }
        float2 *part2 = reinterpret_cast<float2 *>(p.part);
        if (valid) part2[(tm * p.maxseg + seg) * kBM + row] = make_float2(0.0f, dot);
        // the warp that writes the last records of its 32 rows finalises them:
        // n_i = sqrt(max(0, ||W0_i||^2 + 2 s sum dot)), g_i = m_i / n_i
        __threadfence();
        __syncwarp();
        int old = 0;
        if (lane == 0) old = atomicAdd(p.cnt + mt * 4 + quad, 1);
        old = __shfl_sync(0xffffffffu, old, 0);
        int expect = 0;
        for (int c = 0; c < p.nchunks; ++c) {
          const long long ub = (static_cast<long long>(mt) * p.nchunks + c) * p.kbtot;
          expect += cta_of(ub + p.kbtot - 1, p.units, p.ncl) - cta_of(ub, p.units, p.ncl) + 1;
        }
        if (old == expect - 1) {
          __threadfence();
          if (valid) {
            float sd = 0.0f;
            for (int c = 0; c < p.nchunks; ++c) {
              const long long ub = (static_cast<long long>(mt) * p.nchunks + c) * p.kbtot;
              const int nseg = cta_of(ub + p.kbtot - 1, p.units, p.ncl) - cta_of(ub, p.units, p.ncl) + 1;
              const size_t tmc = static_cast<size_t>(mt) * p.nchunks + c;
              for (int j = 0; j < nseg; ++j) sd += __ldcg(part2 + (tmc * p.maxseg + j) * kBM + row).y;
            }
            const float nn = sqrtf(fmaxf(fmaf(p.two_s, sd, p.n0sq[grow]), 0.0f));
            p.norm[grow] = nn;
            p.g[grow] = p.m[grow] / nn;
          }
        }
      } else {
        float *dst = p.part + ((tm * p.maxseg + seg) * kBM + row) * p.NC;
        for (int c = 0; c < p.NC; c += 32) {
          float v[32];
          tmem_ld32(lane_addr + static_cast<uint32_t>(c), v);
          if (valid) {
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
              if (c + j < p.NC) *reinterpret_cast<float4 *>(dst + c + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acce);
      aphase ^= 1u;
      u += kbe - kb0;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem, static_cast<uint32_t>(p.tmem_cols));
  }
}

// ||W0_i||^2 of a bf16 [rows, cols] matrix (cols % 8 == 0): one warp per row,
// lane-strided 128-bit loads, then a fixed shuffle tree
__global__ void __launch_bounds__(256) row_sumsq_bf16_kernel(const __nv_bfloat16 *__restrict__ W, long long rows,
                                                             int cols, float *__restrict__ out) {
  const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const uint4 *w = reinterpret_cast<const uint4 *>(W + row * cols);
  float acc = 0.0f;
  for (int i = lane; i < cols / 8; i += 32) {
    const uint4 q = __ldcs(w + i);
    const uint32_t v[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float lo = __uint_as_float(v[e] << 16), hi = __uint_as_float(v[e] & 0xffff0000u);
      acc = fmaf(lo, lo, acc);
      acc = fmaf(hi, hi, acc);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) out[row] = acc;
}

// B [rows, r] bf16 -> Bp [rows, rp] with zero columns r..rp-1
__global__ void __launch_bounds__(256) pad_cols_bf16_kernel(const __nv_bfloat16 *__restrict__ B, long long rows, int r,
                                                            int rp, __nv_bfloat16 *__restrict__ Bp) {
  const long long n = rows * rp;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const long long row = i / rp;
    const int c = static_cast<int>(i - row * rp);
    Bp[i] = c < r ? B[row * r + c] : __float2bfloat16_rn(0.0f);
  }
}

// (s/2) G from the Gram partial tiles (as gram_reduce_kernel), written as three
// bf16 pieces: g3[a][p * rs + b] for p = 0, 1, 2 with h1 = bf16(v),
// h2 = bf16(v - h1), h3 = bf16(v - h1 - h2); zero outside r (every column
// below rs is written).  Also zeroes the norm pass's ncnt completion counters.
__device__ __forceinline__ void store_g3(int a, int b, float v, int npad, int rs, __nv_bfloat16 *g3) {
  if (a >= npad || b >= rs) return;
  const __nv_bfloat16 h1 = __float2bfloat16_rn(v);
  const float r1 = v - __bfloat162float(h1);
  const __nv_bfloat16 h2 = __float2bfloat16_rn(r1);
  const __nv_bfloat16 h3 = __float2bfloat16_rn(r1 - __bfloat162float(h2));
  __nv_bfloat16 *row = g3 + static_cast<long long>(a) * 3 * rs;
  row[b] = h1;
  row[rs + b] = h2;
  row[2 * rs + b] = h3;
}

__global__ void __launch_bounds__(256) gram_reduce3_kernel(const float *__restrict__ part, StreamK sk, int nchunks,
                                                           int NC, int r, int npad, int rs, float half_s,
                                                           __nv_bfloat16 *__restrict__ g3, int *__restrict__ cnt,
                                                           int ncnt) {
  __shared__ float wsum[8][32][33];
  if (blockIdx.x == 0 && blockIdx.y == 0)
    for (int i = threadIdx.y * 32 + threadIdx.x; i < ncnt; i += 256) cnt[i] = 0;
  const int t = blockIdx.x;
  int mt, nc;
  tile_coords(t, nchunks, 1, &mt, &nc);
  const int nsub = (NC + 31) / 32;
  const int sr = static_cast<int>(blockIdx.y) / nsub, sc = static_cast<int>(blockIdx.y) - sr * nsub;
  const size_t tm = static_cast<size_t>(mt) * nchunks + nc;
  const long long ub = static_cast<long long>(t) * sk.kbtot;
  const int nseg = cta_of(ub + sk.kbtot - 1, sk.units, sk.ncl) - cta_of(ub, sk.units, sk.ncl) + 1;
  const int tx = threadIdx.x, ty = threadIdx.y;
  const int nrow = min(32, min(kBM, r - mt * kBM) - sr * 32);
  const int col = sc * 32 + tx;
  const bool cvalid = col < NC && nc * NC + col < r;
  float acc[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) acc[i] = 0.0f;
  if (cvalid) {
    for (int j = ty; j < nseg; j += 8) {
      const float *pj = part + ((tm * sk.maxseg + j) * kBM + sr * 32) * NC + col;
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (i < nrow) acc[i] += pj[static_cast<size_t>(i) * NC];
    }
  }
#pragma unroll
  for (int i = 0; i < 32; ++i) wsum[ty][i][tx] = acc[i];
  __syncthreads();
  float v[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int i = ty + 8 * q;
    float sum = 0.0f;
#pragma unroll
    for (int w = 0; w < 8; ++w) sum += wsum[w][i][tx];
    v[q] = (i < nrow && cvalid) ? half_s * sum : 0.0f;
  }
  __syncthreads();
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int i = ty + 8 * q;
    store_g3(mt * kBM + sr * 32 + i, nc * NC + col, v[q], npad, rs, g3);
    wsum[0][i][tx] = v[q];
  }
  if (mt != nc) {
    __syncthreads();
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int i = ty + 8 * q;
      store_g3(nc * NC + sc * 32 + i, mt * kBM + sr * 32 + tx, wsum[0][tx][i], npad, rs, g3);
    }
  }
}

// ---------------------------------------------------------------------------
// host planning
// ---------------------------------------------------------------------------
struct GemmPlan {
  TcParams p;
  bool xt;  // M-side operand stored transposed (the kernel instance)
  int bk;   // K indices per K block (the kernel instance): 32 or 64
  size_t smem_bytes;
  size_t part_bytes;
};

int seg_bound(long long units, int ctas, int kbtot) {
  const long long per = units / ctas;  // >= 1 since ctas <= units
  return static_cast<int>((kbtot - 1) / per + 2);
}

// N layout shared by both passes: npad = r rounded to 16, split into equal
// chunks of at most kMaxChunkN.
void plan_n(int r, int *npad, int *nchunks, int *NC) {
  *npad = static_cast<int>(dora::round_up(r, 16));
  *nchunks = static_cast<int>(dora::ceil_div(*npad, kMaxChunkN));
  *NC = static_cast<int>(dora::round_up(dora::ceil_div(*npad, *nchunks), 16));
}

// K = in (+ r for the norm and row passes); at most max_ctas CTAs
bool plan_gemm(int mode, int M, int64_t in, int r, int max_ctas, GemmPlan *gp, int bk = kBK) {
  TcParams &p = gp->p;
  std::memset(&p, 0, sizeof(p));
  gp->xt = false;
  gp->bk = bk;
  p.mode = mode;
  p.M = M;
  int npad;
  plan_n(r, &npad, &p.nchunks, &p.NC);
  if (mode == kGram) {
    // G = A A^T: square 128 x 128 tiles, upper triangle only (M tiles = N chunks)
    p.NC = npad < kBM ? npad : kBM;
    p.nchunks = static_cast<int>(dora::ceil_div(npad, p.NC));
    p.sym = 1;
  }
  const int row_bytes = bk * 4;    // the raw fp32 M-side block
  const int nrow_bytes = bk * 2;   // each bf16 N-side operand
  p.kb1 = static_cast<int>(dora::ceil_div(in, bk));
  p.kbtot = p.kb1 + (mode != kGram ? static_cast<int>(dora::ceil_div(r, bk)) : 0);
  // the N-side tile in nb boxes of nbox rows (a multiple of 8, so every box
  // starts on a swizzle-pattern boundary; at most 256, the box limit)
  p.nb = static_cast<int>(dora::ceil_div(p.NC, 256));
  p.nbox = static_cast<int>(dora::round_up(dora::ceil_div(p.NC, p.nb), 8));
  p.NT = p.nb * p.nbox;
  p.nmma0 = p.NC <= 256 ? p.NC : 256;
  p.nmma1 = p.NC - p.nmma0;
  p.dbl = (mode == kRows && p.nmma1 == 0 && p.NT <= 128) ? 1 : 0;
  // tensor memory: the accumulator (nmma0 columns at 0, nmma1 at 256; with
  // dbl the epilogue also reads 32-column chunks from NT on), then one
  // M-side operand slot per stage (bk columns: bf16 h pairs, then l pairs)
  const int acc_cols = static_cast<int>(p.dbl ? dora::round_up(p.NT + dora::round_up(p.NT, 32), 32)
                                              : dora::round_up(p.nmma1 > 0 ? 256 + p.nmma1 : p.nmma0, 32));
  const int slot_cols = bk;
  p.slot0 = acc_cols;
  // a stage in shared memory: the raw M-side box, then the two N-side tiles
  p.stage_bytes = static_cast<unsigned>(kBM * row_bytes + 2 * p.NT * nrow_bytes);
  p.tx_bytes = p.stage_bytes;
  p.stages = static_cast<int>((kSmemMax - 1024 - 512) / p.stage_bytes);
  if (p.stages > kMaxStages) p.stages = kMaxStages;
  if (p.stages > (512 - acc_cols) / slot_cols) p.stages = (512 - acc_cols) / slot_cols;
  if (p.stages < 2) return false;
  int cols = 32;
  while (cols < acc_cols + p.stages * slot_cols) cols *= 2;
  p.tmem_cols = cols;
  const int mtiles = static_cast<int>(dora::ceil_div(M, kBM));
  p.tiles = p.sym ? p.nchunks * (p.nchunks + 1) / 2 : mtiles * p.nchunks;
  p.units = static_cast<long long>(p.tiles) * p.kbtot;
  const int min_units = mode == kGram ? kMinUnitsGram : kMinUnitsNorm;
  long long ncl = dora::ceil_div(p.units, min_units);
  if (ncl > max_ctas) ncl = max_ctas;
  if (ncl < 1) ncl = 1;
  p.ncl = static_cast<int>(ncl);
  p.ctas = p.ncl;
  p.maxseg = seg_bound(p.units, p.ncl, p.kbtot);
  p.r = r;
  const size_t per_row = mode == kNorm ? 2 : static_cast<size_t>(p.NC);
  gp->part_bytes = static_cast<size_t>(mtiles) * p.nchunks * p.maxseg * kBM * per_row * sizeof(float);
  gp->smem_bytes = static_cast<size_t>(p.stages) * p.stage_bytes + 1024 /*align*/ + 8 * (3 * p.stages + 3) + 64;
  // tensor memory: a CTA holding 512 columns must be alone on its SM
  if (p.tmem_cols > 256 && gp->smem_bytes < 116 * 1024) gp->smem_bytes = 116 * 1024;
  return true;
}

// forward-norm plan: the Gram and norm phases of fwd_norm_kernel
struct FwdPlan {
  FwdParams p;
  size_t smem_bytes;
  size_t part_g_bytes, part_n_bytes;
};

// one phase over M rows (Gram: M = r, N = r; norm: M = out, N = r, K tail r)
void plan_phase(int mode, int M, int64_t in, int r, int fbk, FwdPhase *f, int *mtiles) {
  std::memset(f, 0, sizeof(*f));
  int npad;
  plan_n(r, &npad, &f->nchunks, &f->NC);
  if (mode == kGram) {
    // G = A A^T: square tiles of up to 128 x 128, upper triangle only
    f->NC = npad < kBM ? npad : kBM;
    f->nchunks = static_cast<int>(dora::ceil_div(npad, f->NC));
    f->sym = 1;
  }
  f->kb1 = static_cast<int>(dora::ceil_div(in, fbk));
  f->kbtot = f->kb1 + (mode != kGram ? static_cast<int>(dora::ceil_div(r, fbk)) : 0);
  // N-side TMA boxes of up to 256 rows (the box limit): fewer copies per stage
  f->nb = static_cast<int>(dora::ceil_div(f->NC, 256));
  f->nbox = static_cast<int>(dora::round_up(dora::ceil_div(f->NC, f->nb), 8));
  f->nmma0 = f->NC <= 256 ? f->NC : 256;
  f->nmma1 = f->NC - f->nmma0;
  *mtiles = static_cast<int>(dora::ceil_div(M, kBM));
  f->tiles = f->sym ? f->nchunks * (f->nchunks + 1) / 2 : *mtiles * f->nchunks;
  f->units = static_cast<long long>(f->tiles) * f->kbtot;
}

// Norm-phase CTA boundaries: ub[c] for c = 0 .. C (ub[C] = U), every range
// non-empty, balancing t_unit per unit, t_seg per segment beyond a range's
// first, and t_gram more for the first g CTAs (their Gram phase).  The
// smallest time T at which C ranges cover all units is found by bisection.
void balance_split(long long U, int kbtot, int C, int g, double t_unit, double t_seg, double t_gram,
                   long long *ub) {
  auto fill = [&](double T, bool commit) -> bool {
    long long u = 0;
    for (int c = 0; c < C; ++c) {
      if (commit) ub[c] = u;
      const long long lim = U - (C - 1 - c);   // leave a unit for every later CTA
      double budget = T - (c < g ? t_gram : 0.0);
      const long long start = u;
      while (u < lim) {
        if (u != start && u % kbtot == 0) {   // a new segment
          budget -= t_seg;
          if (budget < t_unit) break;
        }
        long long take = static_cast<long long>(budget / t_unit);
        const long long rem = kbtot - u % kbtot;
        if (take > rem) take = rem;
        if (take > lim - u) take = lim - u;
        if (take <= 0) break;
        u += take;
        budget -= take * t_unit;
      }
      if (u == start) ++u;   // never empty
    }
    if (commit) ub[C] = U;
    return u >= U;
  };
  double lo = U * t_unit / C, hi = lo + t_gram + 2 * t_seg + t_unit;
  while (!fill(hi, false)) hi *= 2;
  for (int it = 0; it < 40; ++it) {
    const double mid = 0.5 * (lo + hi);
    if (fill(mid, false)) hi = mid;
    else lo = mid;
  }
  fill(hi, true);
}

// with_split = false: the geometry and workspace only (no CTA ranges);
// fbk: K indices per K block (32 or 64; 0 = 64 where at least three 64-wide
// stages fit into tensor and shared memory, or two when N is cut into
// several chunks, else 32).  Measured: with N in two chunks of 256 (r = 512)
// 64-wide blocks on two stages take 168 against 172 us; with one chunk of
// 256 (r = 256) 94 against 93
bool plan_fwd(int64_t out, int64_t in, int64_t r, int max_ctas, FwdPlan *fp, bool with_split = true, int fbk = 0) {
  if (fbk == 0) {
    if (plan_fwd(out, in, r, max_ctas, fp, with_split, 64) &&
        (fp->p.S >= 3 || (fp->p.S == 2 && fp->p.ph[1].nchunks > 1)))
      return true;
    return plan_fwd(out, in, r, max_ctas, fp, with_split, 32);
  }
  FwdParams &p = fp->p;
  std::memset(&p, 0, sizeof(p));
  const int ri = static_cast<int>(r);
  p.fbk = fbk;
  const int xbytes = (fbk / kFwdBox) * kFwdBoxBytes;   // one raw-box slot
  const int nrow = fbk * 2;                            // one N-side row of h or l
  int mt_g, mt_n;
  plan_phase(kGram, ri, in, ri, fbk, &p.ph[0], &mt_g);
  plan_phase(kNorm, static_cast<int>(out), in, ri, fbk, &p.ph[1], &mt_n);
  FwdPhase &fg = p.ph[0], &fn = p.ph[1];
  p.M = static_cast<int>(out);
  p.r = ri;
  int nch, NCn;
  plan_n(ri, &p.npad, &nch, &NCn);
  const int nt_g = fg.nb * fg.nbox, nt_n = fn.nb * fn.nbox;
  p.NT = nt_g > nt_n ? nt_g : nt_n;
  p.dbl = (fbk == 64 && fn.nmma1 == 0 && fg.nmma1 == 0 && p.NT <= 64) ? 1 : 0;   // fwd_norm_kernel<64, true>
  // with p.dbl the epilogue reads 32-column chunks at NT on as well
  const int acc_cols = static_cast<int>(
      p.dbl ? dora::round_up(p.NT + dora::round_up(p.NT, 32), 32)
            : dora::round_up(fn.nmma1 > 0 ? 256 + fn.nmma1 : fn.nmma0, 32));
  p.slot0 = acc_cols;
  p.y_bytes = static_cast<unsigned>(p.NT * 2 * nrow);
  // shared memory: as many N-side stages as tensor memory and shared memory
  // allow while leaving at least two more raw-box slots than stages; the rest
  // goes to raw-box slots
  const size_t fixed = 1024 + 8 * (2 * kFwdMaxX + 3 * kFwdMaxS + 7) + 64;
  const size_t budget = kSmemMax - fixed;
  int S = (512 - acc_cols) / fbk;
  if (S > kFwdMaxS) S = kFwdMaxS;
  // raw-box slots: at least two more than stages (one more for 64-wide
  // blocks, whose slots are twice the size)
  const int xspare = fbk == 64 ? 1 : 2;
  while (S >= 2 && static_cast<size_t>(S) * p.y_bytes + static_cast<size_t>(S + xspare) * xbytes > budget) --S;
  if (S < 2) return false;
  int SX = static_cast<int>((budget - static_cast<size_t>(S) * p.y_bytes) / xbytes);
  if (SX > kFwdMaxX) SX = kFwdMaxX;
  p.S = S;
  p.SX = SX;
  int cols = 32;
  while (cols < acc_cols + S * fbk) cols *= 2;
  p.tmem_cols = cols;
  // one CTA per SM, all co-resident: at most max_ctas, at least ... one unit
  // each of the norm phase
  // CTAs: at least four norm units each, at least one per Gram tile (there
  // are never more Gram tiles than norm units), at most one per norm unit
  long long ctas = dora::ceil_div(fn.units, kMinUnitsNorm);
  if (ctas < fg.tiles) ctas = fg.tiles;
  if (ctas > max_ctas) ctas = max_ctas;
  if (ctas > fn.units) ctas = fn.units;
  if (ctas < 1) ctas = 1;
  p.ctas = static_cast<int>(ctas);
  // Cost model measured on GB300: a Gram unit about 0.6 us (latency-bound),
  // a norm unit 0.1 us + 3 N tensor cycles at 1.6 GHz and no less than
  // 0.5 us, a group of reduction loads 1.5 us.
  const double kscale = fbk / 32.0;   // the unit costs below are for 32-wide K blocks
  const double t_norm = std::max(0.5, 0.1 + 3.0 * fn.NC / 1600.0) * kscale;
  // Gram phase: P pieces per tile, one CTA each (the first P * tiles CTAs):
  // about a third of the grid, and enough pieces that the Gram phase takes
  // at most ~35% of a CTA's norm work (s/2 G is needed only after most of it)
  const double t_share = static_cast<double>(fn.units) / p.ctas * t_norm;
  int P = p.ctas / (3 * fg.tiles);
  const int need = static_cast<int>(std::ceil(fg.kbtot * 0.6 * kscale / (0.35 * t_share)));
  if (P < need) P = need;
  if (P > kGramPieces) P = kGramPieces;
  if (P > fg.kbtot) P = fg.kbtot;
  if (P * fg.tiles > p.ctas) P = p.ctas / fg.tiles;
  if (P < 1) return false;   // more Gram tiles than CTAs (not for r <= kMaxR)
  fg.P = P;
  fg.ctas = P * fg.tiles;
  // norm phase: CTA ranges that balance the estimated time per CTA.  Cost
  // model (measured on GB300): a Gram unit 0.75 us; a reduction 1.2 us plus
  // 1.6 us per 32 x 32 block; each segment of a range beyond its first costs
  // an epilogue and the pipeline restart behind it, 1 us + 12.5 us x N / 384
  fn.ctas = p.ctas;
  const int nsub = (fg.NC + 31) / 32;
  const double t_gram =
      fg.kbtot / static_cast<double>(P) * 0.75 * kscale + 1.2 + 1.6 * ((nsub * nsub + P - 1) / P);
  // (with 64-wide K blocks 3 us more: without it, at r = 64 and 128 the
  // CTAs with two segments ended their MMA loops 2.3-2.9 us after the others)
  const double t_seg = 1.0 + 12.5 * fn.NC / 384.0 + (fbk == 64 ? 3.0 : 0.0);
  if (with_split) balance_split(fn.units, fn.kbtot, p.ctas, fg.ctas, t_norm, t_seg, t_gram, p.ub);

  p.nsync = 1 + fg.tiles;
  fp->part_g_bytes = static_cast<size_t>(fg.ctas) * kBM * fg.NC * sizeof(float);
  fp->part_n_bytes = static_cast<size_t>(fn.tiles + p.ctas) * kBM * 2 * sizeof(float);
  fp->smem_bytes = static_cast<size_t>(SX) * xbytes + static_cast<size_t>(S) * p.y_bytes + 1024 +
                   8 * (2 * SX + 3 * S + 7) + 64;
  // the last epilogue's B staging: 4 warps x 32 rows x (N chunk) fp32
  const size_t stage = 4 * static_cast<size_t>((fn.NC + 31) / 32) * 4096;
  p.stage_b = stage <= static_cast<size_t>(SX) * xbytes + static_cast<size_t>(S) * p.y_bytes ? 1 : 0;
  if (p.tmem_cols > 256 && fp->smem_bytes < 116 * 1024) fp->smem_bytes = 116 * 1024;
  return true;
}

cudaError_t launch_fwd(const FwdPlan &fp, cudaStream_t cs, const CUtensorMap &mA, const CUtensorMap &mW0,
                       const CUtensorMap &mB, const CUtensorMap &mAh_g, const CUtensorMap &mAl_g,
                       const CUtensorMap &mAh_n, const CUtensorMap &mAl_n, const CUtensorMap &mGh,
                       const CUtensorMap &mGl, const CUtensorMap &mBs) {
  // CTAs wait on one another (grid-wide counters): a cooperative launch makes
  // them co-resident or fails
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(fp.p.ctas));
  cfg.blockDim = dim3(kFwdThreads);
  cfg.dynamicSmemBytes = fp.smem_bytes;
  cfg.stream = cs;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (fp.p.fbk == 64 && fp.p.dbl)
    return cudaLaunchKernelEx(&cfg, fwd_norm_kernel<64, true>, mA, mW0, mB, mAh_g, mAl_g, mAh_n, mAl_n, mGh, mGl, mBs,
                              fp.p);
  if (fp.p.fbk == 64)
    return cudaLaunchKernelEx(&cfg, fwd_norm_kernel<64>, mA, mW0, mB, mAh_g, mAl_g, mAh_n, mAl_n, mGh, mGl, mBs, fp.p);
  return cudaLaunchKernelEx(&cfg, fwd_norm_kernel<32>, mA, mW0, mB, mAh_g, mAl_g, mAh_n, mAl_n, mGh, mGl, mBs, fp.p);
}

// forward-norm workspace (bf16 three-product scheme): the N-side split of A
// (a_h, a_l: bf16 [r, in8]) and of s/2 G (g_h, g_l: bf16 [npad, npad]), the
// Gram and norm partials, B padded to a 16-byte row when r % 4 != 0, and the
// counters: the fused n / g finalize's [M tiles][4], then the two grid-wide
// phase counters
struct Layout {
  size_t a_h, a_l, g_h, g_l, part_g, part_n, b_pad, cnt, total;
};

size_t al256(size_t x) { return (x + 255) & ~size_t(255); }

// sms: CTAs available
bool plan_layout(int64_t out, int64_t in, int64_t r, int sms, FwdPlan *fp, Layout *L, bool with_split = true) {
  if (!plan_fwd(out, in, r, sms, fp, with_split)) return false;
  int npad, nchunks, NC;
  plan_n(static_cast<int>(r), &npad, &nchunks, &NC);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += al256(bytes);
    return o;
  };
  const size_t in8 = static_cast<size_t>(dora::round_up(in, 8));
  L->a_h = take(static_cast<size_t>(r) * in8 * 2);
  L->a_l = take(static_cast<size_t>(r) * in8 * 2);
  L->g_h = take(static_cast<size_t>(npad) * npad * 2);
  L->g_l = take(static_cast<size_t>(npad) * npad * 2);
  L->part_g = take(fp->part_g_bytes);
  L->part_n = take(fp->part_n_bytes);
  L->b_pad = (r % 4) ? take(static_cast<size_t>(out) * dora::round_up(r, 4) * 4) : 0;
  L->cnt = take((static_cast<size_t>(dora::ceil_div(out, kBM)) * 4 + fp->p.nsync) * sizeof(int));
  L->total = off;
  return true;
}

// gradient through the norm: four GEMM passes and their workspace
struct BwdPlans {
  GemmPlan gg;   // G = A A^T partial tiles (K = in)
  GemmPlan gh;   // s H = B^T (s c (.) B) partial tiles (K = out; B read transposed)
  GemmPlan gb;   // dB rows (M = out, K = in + r)
  GemmPlan ga;   // dA^T rows (M = in, K = out + r; W0 and A read transposed)
  bool small;    // r <= kSgMaxR: G and s H on the CUDA cores (sg) instead of gg, gh
  SgDims sg;
};

// K slices of one Gram product on the CUDA cores: slices of `slice` K indices,
// or longer ones (multiples of the chunk kc) when K would need more than
// `most` of them
void sg_slices(int64_t K, int slice, int kc, int most, int *ns, int *ks) {
  const int64_t n = std::min<int64_t>(dora::ceil_div(K, slice), most);
  const int64_t k = dora::round_up(dora::ceil_div(K, n), kc);
  *ks = static_cast<int>(k);
  *ns = static_cast<int>(dora::ceil_div(K, k));
}
// the N-side operands of the four passes, each a bf16 h / l pair
struct BwdLayout {
  size_t a_h, a_l, y_h, y_l, g_h, g_l, h_h, h_l, part_t, part_r, b_pad, total;
};

bool plan_bwd(int64_t out, int64_t in, int64_t r, int sms, BwdPlans *P, BwdLayout *L) {
  const int ri = static_cast<int>(r);
  if (!plan_gemm(kGram, ri, in, ri, sms, &P->gg)) return false;
  if (!plan_gemm(kGram, ri, out, ri, sms, &P->gh)) return false;
  // the W0 passes: 64-wide K blocks where four stages fit (with three, at
  // r = 128, they measured 4% slower than 32-wide ones), else 32-wide
  auto rows_plan = [&](int M, int64_t K, GemmPlan *gp) {
    if (plan_gemm(kRows, M, K, ri, sms, gp, 64) && gp->p.stages >= 4) return true;
    return plan_gemm(kRows, M, K, ri, sms, gp, 32);
  };
  if (!rows_plan(static_cast<int>(out), in, &P->gb)) return false;
  if (!rows_plan(static_cast<int>(in), out, &P->ga)) return false;
  P->gh.xt = true;
  P->ga.xt = true;
  P->gb.p.chain = kChainK / P->gb.bk;
  P->ga.p.chain = kChainK / P->ga.bk;
  P->small = r <= kSgMaxR;
  SgDims &sg = P->sg;
  std::memset(&sg, 0, sizeof(sg));
  if (P->small) {
    sg.T = r <= 16 ? 16 : r <= 32 ? 32 : 64;
    const int kc = sg.T == 16 ? SgShape<16>::kKC : sg.T == 32 ? SgShape<32>::kKC : SgShape<64>::kKC;
    const int slice = sg.T == 16 ? SgShape<16>::kSlice : sg.T == 32 ? SgShape<32>::kSlice : SgShape<64>::kSlice;
    sg.nt1 = static_cast<int>(dora::ceil_div(r, sg.T));
    sg.ntiles = sg.nt1 * (sg.nt1 + 1) / 2;
    // slices per tile: at most kSgMaxSlices, and no more than the Gram blocks
    // of about one wave (three blocks per SM) need; this also bounds the
    // partials to about 3 * sms tiles
    const int most = std::max(1, std::min(kSgMaxSlices, 3 * sms / (2 * sg.ntiles)));
    sg_slices(in, slice, kc, most, &sg.nsG, &sg.ksG);
    sg_slices(out, slice, kc, most, &sg.nsH, &sg.ksH);
  }
  int npad, nchunks, NC;
  plan_n(ri, &npad, &nchunks, &NC);
  const size_t out8 = static_cast<size_t>(dora::round_up(out, 8));
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += al256(bytes);
    return o;
  };
  const size_t in8 = static_cast<size_t>(dora::round_up(in, 8));
  L->a_h = take(static_cast<size_t>(r) * in8 * 2);     // A: bf16 [r, in8] each
  L->a_l = take(static_cast<size_t>(r) * in8 * 2);
  L->y_h = take(static_cast<size_t>(r) * out8 * 2);    // (s c B)^T: bf16 [r, out8] each
  L->y_l = take(static_cast<size_t>(r) * out8 * 2);
  L->g_h = take(static_cast<size_t>(npad) * npad * 2); // s G: bf16 [npad, npad] each
  L->g_l = take(static_cast<size_t>(npad) * npad * 2);
  L->h_h = take(static_cast<size_t>(npad) * npad * 2); // s^2 H: bf16 [npad, npad] each
  L->h_l = take(static_cast<size_t>(npad) * npad * 2);
  // Gram partials: the CUDA-core slices (small r) or the tensor-core passes' tiles
  L->part_t = take(P->small ? static_cast<size_t>(sg.ntiles) * (sg.nsG + sg.nsH) * sg.T * sg.T * 4
                            : std::max(P->gg.part_bytes, P->gh.part_bytes));
  L->part_r = take(P->gb.part_bytes > P->ga.part_bytes ? P->gb.part_bytes : P->ga.part_bytes);
  L->b_pad = (r % 4) ? take(static_cast<size_t>(out) * dora::round_up(r, 4) * 4) : 0;
  L->total = off;
  return true;
}

bool shape_ok(int64_t out, int64_t in, int64_t r) {
  return out >= 0 && in >= 1 && r >= 1 && r <= kMaxR && out < (1ll << 31) && in < (1ll << 31) &&
         in * r < (1ll << 40);
}

int grid_for(long long n, int sms) {
  long long b = dora::ceil_div(n, 256);
  const long long cap = static_cast<long long>(sms) * 8;
  if (b > cap) b = cap;
  if (b < 1) b = 1;
  return static_cast<int>(b);
}

cudaError_t launch_gemm(const GemmPlan &gp, cudaStream_t cs, const CUtensorMap &x1, const CUtensorMap &x2,
                        const CUtensorMap &y1h, const CUtensorMap &y1l, const CUtensorMap &y2h,
                        const CUtensorMap &y2l) {
  const dim3 grid(static_cast<unsigned>(gp.p.ctas)), block(kThreads);
  const size_t sm = gp.smem_bytes;
#define DORA_TC_LAUNCH(XT_, DBL_, BK_) \
  tc_gemm_kernel<XT_, DBL_, BK_><<<grid, block, sm, cs>>>(x1, x2, y1h, y1l, y2h, y2l, gp.p)
  const bool d = gp.p.dbl != 0;
  if (gp.bk == 64) {
    if (gp.xt) d ? DORA_TC_LAUNCH(true, true, 64) : DORA_TC_LAUNCH(true, false, 64);
    else d ? DORA_TC_LAUNCH(false, true, 64) : DORA_TC_LAUNCH(false, false, 64);
  } else {
    if (gp.xt) d ? DORA_TC_LAUNCH(true, true, 32) : DORA_TC_LAUNCH(true, false, 32);
    else d ? DORA_TC_LAUNCH(false, true, 32) : DORA_TC_LAUNCH(false, false, 32);
  }
#undef DORA_TC_LAUNCH
  return cudaGetLastError();
}

// ---- bf16 weights: planning
struct Plan16 {
  Tc16Params p;
  int bke;   // bf16 per K block (the kernel instance)
  size_t smem_bytes;
  size_t part_bytes;
};

bool plan16(int mode, int M, int64_t in, int r, int max_ctas, Plan16 *gp) {
  Tc16Params &p = gp->p;
  std::memset(&p, 0, sizeof(p));
  p.mode = mode;
  p.M = M;
  int npad;
  plan_n(r, &npad, &p.nchunks, &p.NC);
  if (mode == kGram) {
    p.NC = npad < kBM ? npad : kBM;
    p.nchunks = static_cast<int>(dora::ceil_div(npad, p.NC));
    p.sym = 1;
  }
  p.nb = static_cast<int>(dora::ceil_div(p.NC, 256));   // N-side boxes of up to 256 rows
  p.nbox = static_cast<int>(dora::round_up(dora::ceil_div(p.NC, p.nb), 8));
  p.NT = p.nb * p.nbox;
  p.nmma0 = p.NC <= 256 ? p.NC : 256;
  p.nmma1 = p.NC - p.nmma0;
  const int acc_cols = p.nmma1 > 0 ? 256 + p.nmma1 : p.nmma0;
  int cols = 32;
  while (cols < acc_cols) cols *= 2;
  p.tmem_cols = cols;
  // 64 bf16 per K block (128-byte rows) while a stage fits at least three
  // times into shared memory, else 32 (64-byte rows)
  gp->bke = 0;
  for (int bke = 64; bke >= 32; bke /= 2) {
    const unsigned xb = static_cast<unsigned>(kBM * bke * 2);
    const unsigned sb = xb + static_cast<unsigned>(p.NT * bke * 2);
    const int st = static_cast<int>((kSmemMax - 1024 - 512) / sb);
    if (st >= 3 || bke == 32) {
      gp->bke = bke;
      p.x_bytes = xb;
      p.stage_bytes = sb;
      p.stages = st < kMaxStages ? st : kMaxStages;
      break;
    }
  }
  if (p.stages < 2) return false;
  p.kb1 = static_cast<int>(dora::ceil_div(in, gp->bke));
  p.rs = static_cast<int>(dora::round_up(r, 8));
  p.kbr = static_cast<int>(dora::ceil_div(r, gp->bke));
  p.kbtot = p.kb1 + (mode == kNorm ? 3 * p.kbr : 0);
  const int mtiles = static_cast<int>(dora::ceil_div(M, kBM));
  p.tiles = p.sym ? p.nchunks * (p.nchunks + 1) / 2 : mtiles * p.nchunks;
  p.units = static_cast<long long>(p.tiles) * p.kbtot;
  const int min_units = mode == kGram ? kMinUnitsGram : kMinUnitsNorm;
  long long ncl = dora::ceil_div(p.units, min_units);
  if (ncl > max_ctas) ncl = max_ctas;
  if (ncl < 1) ncl = 1;
  p.ncl = static_cast<int>(ncl);
  p.ctas = p.ncl;
  p.maxseg = seg_bound(p.units, p.ncl, p.kbtot);
  p.r = r;
  const size_t per_row = mode == kGram ? static_cast<size_t>(p.NC) : 2;
  gp->part_bytes = static_cast<size_t>(mtiles) * p.nchunks * p.maxseg * kBM * per_row * sizeof(float);
  gp->smem_bytes = static_cast<size_t>(p.stages) * p.stage_bytes + 1024 /*align*/ + 8 * (2 * p.stages + 3) + 64;
  if (p.tmem_cols > 256 && gp->smem_bytes < 116 * 1024) gp->smem_bytes = 116 * 1024;
  return true;
}

struct Layout16 {
  size_t g3, part_g, part_n, b_pad, cnt, total;
};

bool plan_layout16(int64_t out, int64_t in, int64_t r, int sms, Plan16 *gg, Plan16 *gn, Layout16 *L) {
  if (!plan16(kGram, static_cast<int>(r), in, static_cast<int>(r), sms, gg)) return false;
  if (!plan16(kNorm, static_cast<int>(out), in, static_cast<int>(r), sms, gn)) return false;
  int npad, nchunks, NC;
  plan_n(static_cast<int>(r), &npad, &nchunks, &NC);
  const int64_t rs = dora::round_up(r, 8);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += al256(bytes);
    return o;
  };
  L->g3 = take(static_cast<size_t>(npad) * 3 * rs * 2);
  L->part_g = take(gg->part_bytes);
  L->part_n = take(gn->part_bytes);
  L->b_pad = (r % 8) ? take(static_cast<size_t>(out) * rs * 2) : 0;
  L->cnt = take(static_cast<size_t>(dora::ceil_div(out, kBM)) * 4 * sizeof(int));
  L->total = off;
  return true;
}

cudaError_t launch16(const Plan16 &gp, cudaStream_t cs, const CUtensorMap &x1, const CUtensorMap &x2,
                     const CUtensorMap &y1, const CUtensorMap &y2) {
  const dim3 grid(static_cast<unsigned>(gp.p.ctas)), block(kThreads);
  if (gp.bke == 64)
    tc16_kernel<64><<<grid, block, gp.smem_bytes, cs>>>(x1, x2, y1, y2, gp.p);
  else
    tc16_kernel<32><<<grid, block, gp.smem_bytes, cs>>>(x1, x2, y1, y2, gp.p);
  return cudaGetLastError();
}

// Once per device and context: the address of the device error word and the
// shared-memory limit of every tensor-core kernel instance.
dora_status device_init(int device, int **errp) {
  static std::mutex mu;
  static int *err_ptr[64] = {};
  static uint64_t ctx_of[64] = {};
  std::lock_guard<std::mutex> lock(mu);
  if (device < 0 || device >= 64) return DORA_ERR_CUDA;
  const uint64_t ctx = dora::context_id();
  if (!err_ptr[device] || ctx == 0 || ctx != ctx_of[device]) {
    err_ptr[device] = nullptr;
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_dora_err) != cudaSuccess) return DORA_ERR_CUDA;
    const cudaFuncAttribute a = cudaFuncAttributeMaxDynamicSharedMemorySize;
    if (cudaFuncSetAttribute(tc_gemm_kernel<false>, a, kSmemMax) != cudaSuccess ||
        cudaFuncSetAttribute(tc_gemm_kernel<true>, a, kSmemMax) != cudaSuccess ||
        cudaFuncSetAttribute(tc_gemm_kernel<false, true>, a, kSmemMax) != cudaSuccess ||
        cudaFuncSetAttribute(tc_gemm_kernel<true, true>, a, kSmemMax) != cudaSuccess ||
        cudaFuncSetAttribute(tc_gemm_kernel<false, false, 64>, a, kSmemMax) != cudaSuccess ||
        cudaFuncSetAttribute(tc_gemm_kernel<true, false, 64>, a, kSmemMax) != cudaSuccess ||
        cudaFuncSetAttribute(tc_gemm_kernel<false, true, 64>, a, kSmemMax) != cudaSuccess ||
        cudaFuncSetAttribute(tc_gemm_kernel<true, true, 64>, a, kSmemMax) != cudaSuccess ||
        cudaFuncSetAttribute(fwd_norm_kernel<32>, a, kSmemMax) != cudaSuccess ||
        cudaFuncSetAttribute(fwd_norm_kernel<64>, a, kSmemMax) != cudaSuccess ||
        cudaFuncSetAttribute(fwd_norm_kernel<64, true>, a, kSmemMax) != cudaSuccess ||
        cudaFuncSetAttribute(tc16_kernel<32>, a, kSmemMax) != cudaSuccess ||
        cudaFuncSetAttribute(tc16_kernel<64>, a, kSmemMax) != cudaSuccess)
      return DORA_ERR_CUDA;
    err_ptr[device] = static_cast<int *>(ptr);
    ctx_of[device] = dora::context_id();
  }
  *errp = err_ptr[device];
  return DORA_OK;
}

}  // namespace

namespace dora {
dora_status error_word(int device, int **errp) { return device_init(device, errp); }
dora_status test_hooks(int **stall, unsigned long long **limit_ns) {
  void *a = nullptr, *b = nullptr;
  if (cudaGetSymbolAddress(&a, g_dora_stall) != cudaSuccess ||
      cudaGetSymbolAddress(&b, g_wait_limit_ns) != cudaSuccess)
    return DORA_ERR_CUDA;
  *stall = static_cast<int *>(a);
  *limit_ns = static_cast<unsigned long long *>(b);
  return DORA_OK;
}
}  // namespace dora

extern "C" size_t dora_norm_factored_workspace(int64_t out, int64_t in, int64_t r) {
  if (!shape_ok(out, in, r)) return 0;
  // the layout for kMaxCtas CTAs: the partial-result space only grows with
  // the CTA count, so this bounds every device with up to kMaxCtas SMs
  FwdPlan fp;
  Layout L;
  if (!plan_layout(out > 0 ? out : 1, in, r, kMaxCtas, &fp, &L, false)) return 0;
  return L.total;
}

extern "C" dora_status dora_test_stall_loads(int on, uint64_t wait_limit_ns) {
  const int v = on ? 1 : 0;
  const unsigned long long lim = wait_limit_ns ? wait_limit_ns : kWaitLimitNs;
  if (cudaMemcpyToSymbol(g_dora_stall, &v, sizeof(v)) != cudaSuccess ||
      cudaMemcpyToSymbol(g_wait_limit_ns, &lim, sizeof(lim)) != cudaSuccess)
    return DORA_ERR_CUDA;
  return DORA_OK;
}

extern "C" dora_status dora_device_error(int *code) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_dora_err, sizeof(int)) != cudaSuccess) return DORA_ERR_CUDA;
  if (code) *code = v;
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_dora_err, &zero, sizeof(int)) != cudaSuccess) return DORA_ERR_CUDA;
    return DORA_ERR_DEVICE;
  }
  return DORA_OK;
}

namespace {
// Host-side caches of the forward norm, so that repeated calls (a training
// loop calls it with the same shapes and, mostly, the same buffers every
// step) skip the planning and the tensor-map encoding:
//   plans  per (device, out, in, r): the phase geometry, the balanced CTA
//          ranges and the workspace layout;
//   maps   per (device, W0, A, B, workspace, out, in, r): the ten encoded
//          tensor maps (they hold these addresses).
// Both are small rings of entries; a miss recomputes and replaces the oldest.
constexpr int kCacheEntries = 8;
struct PlanEntry {
  bool used;
  int device, sms;
  int64_t out, in, r;
  FwdPlan fp;
  Layout L;
};
struct MapEntry {
  bool used;
  int device;
  const void *W0, *A, *B, *ws;
  int64_t out, in, r;
  CUtensorMap maps[10];
};
std::mutex g_cache_mu;
PlanEntry g_plans[kCacheEntries];
MapEntry g_maps[kCacheEntries];
int g_plan_next = 0, g_map_next = 0;

bool cached_plan(int device, int sms, int64_t out, int64_t in, int64_t r, FwdPlan *fp, Layout *L) {
  {
    std::lock_guard<std::mutex> lock(g_cache_mu);
    for (const PlanEntry &e : g_plans)
      if (e.used && e.device == device && e.sms == sms && e.out == out && e.in == in && e.r == r) {
        *fp = e.fp;
        *L = e.L;
        return true;
      }
  }
  if (!plan_layout(out, in, r, sms, fp, L)) return false;
  std::lock_guard<std::mutex> lock(g_cache_mu);
  PlanEntry &e = g_plans[g_plan_next];
  g_plan_next = (g_plan_next + 1) % kCacheEntries;
  e.used = true;
  e.device = device;
  e.sms = sms;
  e.out = out;
  e.in = in;
  e.r = r;
  e.fp = *fp;
  e.L = *L;
  return true;
}

bool find_maps(int device, const void *W0, const void *A, const void *B, const void *ws, int64_t out, int64_t in,
               int64_t r, CUtensorMap *maps) {
  std::lock_guard<std::mutex> lock(g_cache_mu);
  for (const MapEntry &e : g_maps)
    if (e.used && e.device == device && e.W0 == W0 && e.A == A && e.B == B && e.ws == ws && e.out == out &&
        e.in == in && e.r == r) {
      std::memcpy(maps, e.maps, sizeof(e.maps));
      return true;
    }
  return false;
}

void keep_maps(int device, const void *W0, const void *A, const void *B, const void *ws, int64_t out, int64_t in,
               int64_t r, const CUtensorMap *maps) {
  std::lock_guard<std::mutex> lock(g_cache_mu);
  MapEntry &e = g_maps[g_map_next];
  g_map_next = (g_map_next + 1) % kCacheEntries;
  e.used = true;
  e.device = device;
  e.W0 = W0;
  e.A = A;
  e.B = B;
  e.ws = ws;
  e.out = out;
  e.in = in;
  e.r = r;
  std::memcpy(e.maps, maps, sizeof(e.maps));
}
}  // namespace

extern "C" dora_status dora_norm_factored(const float *W0, const float *A, const float *B, const float *m, float s,
                                          int64_t out, int64_t in, int64_t r, float *norm, float *g,
                                          void *workspace, size_t workspace_bytes, dora_stream_t stream) {
  if (!shape_ok(out, in, r)) return DORA_ERR_SHAPE;
  if (out == 0) return DORA_OK;
  if (!W0 || !A || !B || !m || !norm || !g) return DORA_ERR_NULL;
  if (!workspace) return DORA_ERR_WORKSPACE;
  if (in % 4 != 0) return DORA_ERR_ALIGN;
  if (!dora::aligned(W0, 16) || !dora::aligned(A, 16) || !dora::aligned(B, 16) || !dora::aligned(m, 4) ||
      !dora::aligned(norm, 4) || !dora::aligned(g, 4))
    return DORA_ERR_ALIGN;
  if (!dora::aligned(workspace, 256) || workspace_bytes < dora_norm_factored_workspace(out, in, r))
    return DORA_ERR_WORKSPACE;

  dora::DeviceInfo info;
  int device = 0;
  dora_status st = dora::current_device(&info, &device);
  if (st != DORA_OK) return st;
  const int sms = info.sms < kMaxCtas ? info.sms : kMaxCtas;

  int *errp = nullptr;
  st = device_init(device, &errp);
  if (st != DORA_OK) return st;

  FwdPlan fp;
  Layout L;
  if (!cached_plan(device, sms, out, in, r, &fp, &L)) return DORA_ERR_SHAPE;
  if (workspace_bytes < L.total) return DORA_ERR_WORKSPACE;   // never: the size above bounds every device
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  __nv_bfloat16 *a_h = reinterpret_cast<__nv_bfloat16 *>(ws + L.a_h);
  __nv_bfloat16 *a_l = reinterpret_cast<__nv_bfloat16 *>(ws + L.a_l);
  const float *Bk = B;
  int64_t ldb = r;
  const int npad = fp.p.npad;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  uint64_t launches = 0;

  // 1. N-side split of A (bf16 h and l) and zero counters; B padded to a
  //    TMA-legal row stride when r % 4 != 0
  const int in8 = static_cast<int>(dora::round_up(in, 8));
  int *cnt = reinterpret_cast<int *>(ws + L.cnt);
  const int ncnt = static_cast<int>(dora::ceil_div(out, kBM)) * 4;
  split_hl_kernel<<<grid_for(r * in8 / 4, sms), 256, 0, cs>>>(A, r, static_cast<int>(in), in8, a_h, a_l, cnt,
                                                               ncnt + fp.p.nsync);
  ++launches;
  if (r % 4) {
    const int rp = static_cast<int>(dora::round_up(r, 4));
    float *bp = reinterpret_cast<float *>(ws + L.b_pad);
    pad_cols_kernel<<<grid_for(out * rp, sms), 256, 0, cs>>>(B, out, static_cast<int>(r), rp, bp);
    ++launches;
    Bk = bp;
    ldb = rp;
  }

  // tensor maps: the raw fp32 M-side boxes are 128 x 32 (128-byte rows), the
  // bf16 N-side boxes nbox x 32 (64-byte rows); the N-side boxes of the two
  // phases may differ in height, so one map set each
  FwdParams &p = fp.p;
  p.ph[0].part = reinterpret_cast<float *>(ws + L.part_g);
  p.ph[1].part = reinterpret_cast<float *>(ws + L.part_n);
  p.err = errp;
  p.cnt = cnt;
  p.sync = cnt + ncnt;
  p.m = m;
  p.norm = norm;
  p.g = g;
  p.two_s = 2.0f * s;
  p.half_s = 0.5f * s;
  p.Bk = Bk;
  p.ldb = static_cast<int>(ldb);
  p.gs_h = reinterpret_cast<__nv_bfloat16 *>(ws + L.g_h);
  p.gs_l = reinterpret_cast<__nv_bfloat16 *>(ws + L.g_l);
  // map order: A, Ah_g, Al_g, Ah_n, Al_n, W0, B, Gh, Gl, B staging
  CUtensorMap mp[10];
  if (!find_maps(device, W0, A, B, workspace, out, in, r, mp)) {
    const int nbg = p.ph[0].nbox, nbn = p.ph[1].nbox;
    const int yb = 2 * p.fbk;   // bytes of an N-side box row (one K block of bf16)
    const bool ok =
        make_map(&mp[0], A, false, r, in, in, kBM, 128) && make_map(&mp[1], a_h, true, r, in8, in8, nbg, yb) &&
        make_map(&mp[2], a_l, true, r, in8, in8, nbg, yb) && make_map(&mp[3], a_h, true, r, in8, in8, nbn, yb) &&
        make_map(&mp[4], a_l, true, r, in8, in8, nbn, yb) && make_map(&mp[5], W0, false, out, in, in, kBM, 128) &&
        make_map(&mp[6], Bk, false, out, ldb, ldb, kBM, 128) &&
        make_map(&mp[7], p.gs_h, true, npad, npad, npad, nbn, yb) &&
        make_map(&mp[8], p.gs_l, true, npad, npad, npad, nbn, yb) &&
        make_map(&mp[9], Bk, false, out, ldb, ldb, 32, 128);   // 32 x 32 boxes for the B staging
    if (!ok) {
      dora::count_launches(launches);
      return DORA_ERR_CUDA;
    }
    keep_maps(device, W0, A, B, workspace, out, in, r, mp);
  }

  // 2. one launch: Gram partials, the reduction into s/2 G (split), and
  //    [W0 | B] x [A | s/2 G]^T with per-segment row reductions; the last
  //    epilogue warp of each quarter M tile writes n and g
  if (launch_fwd(fp, cs, mp[0], mp[5], mp[6], mp[1], mp[2], mp[3], mp[4], mp[7], mp[8], mp[9]) != cudaSuccess) {
    dora::count_launches(launches);
    return DORA_ERR_CUDA;
  }
  ++launches;
  dora::count_launches(launches);
  return dora::launch_status();
}

// ---------------------------------------------------------------------------
// gradient through the norm
// ---------------------------------------------------------------------------
extern "C" size_t dora_norm_factored_bwd_workspace(int64_t out, int64_t in, int64_t r) {
  if (!shape_ok(out, in, r)) return 0;
  BwdPlans P;
  BwdLayout L;
  if (!plan_bwd(out > 0 ? out : 1, in, r, kMaxCtas, &P, &L)) return 0;
  return L.total;
}

extern "C" dora_status dora_norm_factored_bwd(const float *W0, const float *A, const float *B, const float *norm,
                                              const float *g, const float *d_mag, float s, int64_t out, int64_t in,
                                              int64_t r, float *dA, float *dB, void *workspace,
                                              size_t workspace_bytes, dora_stream_t stream) {
  if (!shape_ok(out, in, r)) return DORA_ERR_SHAPE;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (out == 0) {
    // no rows: dA is an empty sum and dB has no elements
    if (!dA) return DORA_ERR_NULL;
    if (!dora::aligned(dA, 4)) return DORA_ERR_ALIGN;
    if (cudaMemsetAsync(dA, 0, static_cast<size_t>(r) * in * sizeof(float), cs) != cudaSuccess) return DORA_ERR_CUDA;
    return DORA_OK;
  }
  if (!W0 || !A || !B || !norm || !g || !d_mag || !dA || !dB) return DORA_ERR_NULL;
  if (!workspace) return DORA_ERR_WORKSPACE;
  if (in % 4 != 0) return DORA_ERR_ALIGN;
  if (!dora::aligned(W0, 16) || !dora::aligned(A, 16) || !dora::aligned(B, 16) || !dora::aligned(norm, 4) ||
      !dora::aligned(g, 4) || !dora::aligned(d_mag, 4) || !dora::aligned(dA, 4) || !dora::aligned(dB, 4))
    return DORA_ERR_ALIGN;
  if (!dora::aligned(workspace, 256) || workspace_bytes < dora_norm_factored_bwd_workspace(out, in, r))
    return DORA_ERR_WORKSPACE;

  dora::DeviceInfo info;
  int device = 0;
  dora_status st = dora::current_device(&info, &device);
  if (st != DORA_OK) return st;
  const int sms = info.sms < kMaxCtas ? info.sms : kMaxCtas;
  int *errp = nullptr;
  st = device_init(device, &errp);
  if (st != DORA_OK) return st;

  BwdPlans P;
  BwdLayout L;
  if (!plan_bwd(out, in, r, sms, &P, &L)) return DORA_ERR_SHAPE;
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  auto bf = [&](size_t o) { return reinterpret_cast<__nv_bfloat16 *>(ws + o); };
  __nv_bfloat16 *a_h = bf(L.a_h), *a_l = bf(L.a_l), *y_h = bf(L.y_h), *y_l = bf(L.y_l);
  __nv_bfloat16 *g_h = bf(L.g_h), *g_l = bf(L.g_l), *h_h = bf(L.h_h), *h_l = bf(L.h_l);
  float *part_t = reinterpret_cast<float *>(ws + L.part_t);
  float *part_r = reinterpret_cast<float *>(ws + L.part_r);
  int npad, nchunks, NC;
  plan_n(static_cast<int>(r), &npad, &nchunks, &NC);
  const int64_t in8 = dora::round_up(in, 8), out8 = dora::round_up(out, 8);
  uint64_t launches = 0;
  auto fail = [&]() {
    dora::count_launches(launches);
    return DORA_ERR_CUDA;
  };

  // 1. B padded to a TMA-legal row stride when r % 4 != 0; then one launch:
  //    the N-side splits of A and of (s c B)^T and, for r <= kSgMaxR, the
  //    partials of G and s H
  const float *Bk = B;
  int64_t ldb = r;
  if (r % 4) {
    const int rp = static_cast<int>(dora::round_up(r, 4));
    float *bp = reinterpret_cast<float *>(ws + L.b_pad);
    pad_cols_kernel<<<grid_for(out * rp, sms), 256, 0, cs>>>(B, out, static_cast<int>(r), rp, bp);
    ++launches;
    Bk = bp;
    ldb = rp;
  }
  {
    GradPrep gp;
    gp.sg = P.sg;
    gp.nb_sg = P.small ? P.sg.ntiles * (P.sg.nsG + P.sg.nsH) : 0;
    gp.bs_bx = static_cast<int>(dora::ceil_div(out8, 32));
    gp.nb_bs = gp.bs_bx * static_cast<int>(dora::ceil_div(r, kBsCols));
    gp.nb_split = grid_for(r * in8 / 4, sms);
    gp.A = A;
    gp.r = static_cast<int>(r);
    gp.in = static_cast<int>(in);
    gp.in8 = static_cast<int>(in8);
    gp.a_h = a_h;
    gp.a_l = a_l;
    gp.B = B;
    gp.out = out;
    gp.out8 = out8;
    gp.g = g;
    gp.d_mag = d_mag;
    gp.norm = norm;
    gp.s = s;
    gp.y_h = y_h;
    gp.y_l = y_l;
    gp.sg_part = part_t;
    const unsigned nblk = static_cast<unsigned>(gp.nb_sg + gp.nb_bs + gp.nb_split);
    switch (P.sg.T) {
      case 16: grad_prep_kernel<16><<<nblk, 256, 0, cs>>>(gp); break;
      case 32: grad_prep_kernel<32><<<nblk, 256, 0, cs>>>(gp); break;
      case 64: grad_prep_kernel<64><<<nblk, 256, 0, cs>>>(gp); break;
      default: grad_prep_kernel<0><<<nblk, 256, 0, cs>>>(gp); break;
    }
    ++launches;
  }

  // tensor maps: the raw fp32 M-side boxes (one K block of 32 by 128 rows) and
  // the bf16 N-side boxes (64-byte rows of 32 K indices)
  const GemmPlan &gg = P.gg, &gh = P.gh, &gb = P.gb, &ga = P.ga;
  // raw fp32 boxes of 32 K (128-byte rows); N-side rows of each pass's K block
  const int rb = 4 * kBK, nb = 2 * kBK, nbb = 2 * gb.bk, nba = 2 * ga.bk;
  CUtensorMap mA, mAh_g, mAl_g, mBt, mYh_h, mYl_h, mW0, mB, mAh_b, mAl_b, mGh, mGl, mW0t, mAt, mYh_a, mYl_a, mHh, mHl;
  bool ok = make_map(&mW0, W0, false, out, in, in, kBM, rb) && make_map(&mB, Bk, false, out, ldb, ldb, kBM, rb) &&
            make_map(&mAh_b, a_h, true, r, in8, in8, gb.p.nbox, nbb) &&
            make_map(&mAl_b, a_l, true, r, in8, in8, gb.p.nbox, nbb) &&
            make_map(&mGh, g_h, true, npad, npad, npad, gb.p.nbox, nbb) &&
            make_map(&mGl, g_l, true, npad, npad, npad, gb.p.nbox, nbb) &&
            make_map_t(&mW0t, W0, out, in, in, ga.bk) && make_map_t(&mAt, A, r, in, in, ga.bk) &&
            make_map(&mYh_a, y_h, true, r, out8, out8, ga.p.nbox, nba) &&
            make_map(&mYl_a, y_l, true, r, out8, out8, ga.p.nbox, nba) &&
            make_map(&mHh, h_h, true, npad, npad, npad, ga.p.nbox, nba) &&
            make_map(&mHl, h_l, true, npad, npad, npad, ga.p.nbox, nba);
  if (ok && !P.small)
    ok = make_map(&mA, A, false, r, in, in, kBM, rb) && make_map(&mAh_g, a_h, true, r, in8, in8, gg.p.nbox, nb) &&
         make_map(&mAl_g, a_l, true, r, in8, in8, gg.p.nbox, nb) && make_map_t(&mBt, Bk, out, r, ldb, kBK) &&
         make_map(&mYh_h, y_h, true, r, out8, out8, gh.p.nbox, nb) &&
         make_map(&mYl_h, y_l, true, r, out8, out8, gh.p.nbox, nb);
  if (!ok) return fail();

  if (P.small) {
    // 2-3. s G and s^2 H from the partials (fixed-order sums, split)
    sg_fin_kernel<<<2 * P.sg.ntiles * (P.sg.T * P.sg.T / 64), 256, 0, cs>>>(part_t, P.sg, npad, s, g_h, g_l, h_h,
                                                                              h_l);
    ++launches;
  } else {
    // 2. s G = s A A^T (partial tiles, fixed-order reduction, split)
    GemmPlan pg = gg;
    pg.p.part = part_t;
    pg.p.err = errp;
    if (launch_gemm(pg, cs, mA, mA, mAh_g, mAl_g, mAh_g, mAl_g) != cudaSuccess) return fail();
    ++launches;
    {
      const StreamK sk{pg.p.units, pg.p.ncl, pg.p.kbtot, pg.p.maxseg};
      const int nsub = (pg.p.NC + 31) / 32;
      gram_reduce_kernel<<<dim3(static_cast<unsigned>(pg.p.tiles), static_cast<unsigned>(nsub * nsub)),
                                 dim3(32, 8), 0, cs>>>(part_t, sk, pg.p.nchunks, pg.p.NC, static_cast<int>(r), npad,
                                                       s, g_h, g_l);
      ++launches;
    }
    // 3. s^2 H = s (B^T (s c (.) B)), B read transposed
    GemmPlan ph = gh;
    ph.p.part = part_t;
    ph.p.err = errp;
    if (launch_gemm(ph, cs, mBt, mBt, mYh_h, mYl_h, mYh_h, mYl_h) != cudaSuccess) return fail();
    ++launches;
    {
      const StreamK sk{ph.p.units, ph.p.ncl, ph.p.kbtot, ph.p.maxseg};
      const int nsub = (ph.p.NC + 31) / 32;
      gram_reduce_kernel<<<dim3(static_cast<unsigned>(ph.p.tiles), static_cast<unsigned>(nsub * nsub)),
                                 dim3(32, 8), 0, cs>>>(part_t, sk, ph.p.nchunks, ph.p.NC, static_cast<int>(r), npad,
                                                       s, h_h, h_l);
      ++launches;
    }
  }
  // 4. dB = s c (.) ([W0 | B] x [A | s G]^T): partial rows, then their sum
  GemmPlan pb = gb;
  pb.p.part = part_r;
  pb.p.err = errp;
  if (launch_gemm(pb, cs, mW0, mB, mAh_b, mAl_b, mGh, mGl) != cudaSuccess) return fail();
  ++launches;
  {
    const StreamK sk{pb.p.units, pb.p.ncl, pb.p.kbtot, pb.p.maxseg};
    const unsigned mtiles = static_cast<unsigned>(dora::ceil_div(out, kBM));
    rows_reduce_kernel<<<dim3(mtiles * pb.p.nchunks, static_cast<unsigned>((pb.p.NC + 31) / 32)), 256, 0, cs>>>(
        reinterpret_cast<const float4 *>(part_r), sk, pb.p.nchunks, pb.p.NC, static_cast<int>(out),
        static_cast<int>(r), 0, g, d_mag, norm, s, dB, r);
    ++launches;
  }
  // 5. dA^T = [W0^T | A^T] x [(s c B)^T | s^2 H]^T, summed and written
  //    transposed into dA
  GemmPlan pa = ga;
  pa.p.part = part_r;
  pa.p.err = errp;
  if (launch_gemm(pa, cs, mW0t, mAt, mYh_a, mYl_a, mHh, mHl) != cudaSuccess) return fail();
  ++launches;
  {
    const StreamK sk{pa.p.units, pa.p.ncl, pa.p.kbtot, pa.p.maxseg};
    const unsigned mtiles = static_cast<unsigned>(dora::ceil_div(in, kBM));
    rows_reduce_kernel<<<dim3(mtiles * pa.p.nchunks, static_cast<unsigned>((pa.p.NC + 31) / 32)), 256, 0, cs>>>(
        reinterpret_cast<const float4 *>(part_r), sk, pa.p.nchunks, pa.p.NC, static_cast<int>(in),
        static_cast<int>(r), 1, g, d_mag, norm, s, dA, in);
    ++launches;
  }
  dora::count_launches(launches);
  return dora::launch_status();
}

// ---------------------------------------------------------------------------
// bf16 weights
// ---------------------------------------------------------------------------
extern "C" size_t dora_norm_factored_bf16_workspace(int64_t out, int64_t in, int64_t r) {
  if (!shape_ok(out, in, r)) return 0;
  Plan16 gg, gn;
  Layout16 L;
  if (!plan_layout16(out > 0 ? out : 1, in, r, kMaxCtas, &gg, &gn, &L)) return 0;
  return L.total;
}

extern "C" dora_status dora_row_sumsq_bf16(const void *W0, int64_t rows, int64_t cols, float *n0sq,
                                           dora_stream_t stream) {
  if (rows < 0 || cols < 1 || rows >= (1ll << 31) || cols >= (1ll << 31)) return DORA_ERR_SHAPE;
  if (rows == 0) return DORA_OK;
  if (!W0 || !n0sq) return DORA_ERR_NULL;
  if (cols % 8 != 0 || !dora::aligned(W0, 16) || !dora::aligned(n0sq, 4)) return DORA_ERR_ALIGN;
  dora::DeviceInfo info;
  int device = 0;
  dora_status st = dora::current_device(&info, &device);
  if (st != DORA_OK) return st;
  row_sumsq_bf16_kernel<<<static_cast<unsigned>(dora::ceil_div(rows, 8)), 256, 0,
                          reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<const __nv_bfloat16 *>(W0), rows, static_cast<int>(cols), n0sq);
  dora::count_launches(1);
  return dora::launch_status();
}

extern "C" dora_status dora_norm_factored_bf16(const void *W0, const void *A, const void *B, const float *m,
                                               const float *n0sq, float s, int64_t out, int64_t in, int64_t r,
                                               float *norm, float *g, void *workspace, size_t workspace_bytes,
                                               dora_stream_t stream) {
  if (!shape_ok(out, in, r)) return DORA_ERR_SHAPE;
  if (out == 0) return DORA_OK;
  if (!W0 || !A || !B || !m || !n0sq || !norm || !g) return DORA_ERR_NULL;
  if (!workspace) return DORA_ERR_WORKSPACE;
  if (in % 8 != 0) return DORA_ERR_ALIGN;
  if (!dora::aligned(W0, 16) || !dora::aligned(A, 16) || !dora::aligned(B, 16) || !dora::aligned(m, 4) ||
      !dora::aligned(n0sq, 4) || !dora::aligned(norm, 4) || !dora::aligned(g, 4))
    return DORA_ERR_ALIGN;
  if (!dora::aligned(workspace, 256) || workspace_bytes < dora_norm_factored_bf16_workspace(out, in, r))
    return DORA_ERR_WORKSPACE;

  dora::DeviceInfo info;
  int device = 0;
  dora_status st = dora::current_device(&info, &device);
  if (st != DORA_OK) return st;
  const int sms = info.sms < kMaxCtas ? info.sms : kMaxCtas;
  int *errp = nullptr;
  st = device_init(device, &errp);
  if (st != DORA_OK) return st;

  Plan16 gg, gn;
  Layout16 L;
  if (!plan_layout16(out, in, r, sms, &gg, &gn, &L)) return DORA_ERR_SHAPE;
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  __nv_bfloat16 *g3 = reinterpret_cast<__nv_bfloat16 *>(ws + L.g3);
  float *part_g = reinterpret_cast<float *>(ws + L.part_g);
  float *part_n = reinterpret_cast<float *>(ws + L.part_n);
  int *cnt = reinterpret_cast<int *>(ws + L.cnt);
  const int ncnt = static_cast<int>(dora::ceil_div(out, kBM)) * 4;
  int npad, nchunks, NC;
  plan_n(static_cast<int>(r), &npad, &nchunks, &NC);
  const int64_t rs = dora::round_up(r, 8);
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  uint64_t launches = 0;

  // B padded to a 16-byte row when r % 8 != 0
  const __nv_bfloat16 *Bk = static_cast<const __nv_bfloat16 *>(B);
  int64_t ldb = r;
  if (r % 8) {
    __nv_bfloat16 *bp = reinterpret_cast<__nv_bfloat16 *>(ws + L.b_pad);
    pad_cols_bf16_kernel<<<grid_for(out * rs, sms), 256, 0, cs>>>(Bk, out, static_cast<int>(r), static_cast<int>(rs),
                                                                  bp);
    ++launches;
    Bk = bp;
    ldb = rs;
  }

  // tensor maps (box rows: one K block of bf16, 64 or 128 bytes)
  CUtensorMap mAx, mAy_g, mW0, mAy_n, mB, mG3;
  const int rbg = 2 * gg.bke, rbn = 2 * gn.bke;
  bool ok = make_map(&mAx, A, true, r, in, in, kBM, rbg) && make_map(&mAy_g, A, true, r, in, in, gg.p.nbox, rbg) &&
            make_map(&mW0, W0, true, out, in, in, kBM, rbn) && make_map(&mAy_n, A, true, r, in, in, gn.p.nbox, rbn) &&
            make_map(&mB, Bk, true, out, ldb, ldb, kBM, rbn) &&
            make_map(&mG3, g3, true, npad, 3 * rs, 3 * rs, gn.p.nbox, rbn);
  if (!ok) {
    dora::count_launches(launches);
    return DORA_ERR_CUDA;
  }

  // 1. Gram partial tiles
  gg.p.part = part_g;
  gg.p.err = errp;
  if (launch16(gg, cs, mAx, mAx, mAy_g, mAy_g) != cudaSuccess) {
    dora::count_launches(launches);
    return DORA_ERR_CUDA;
  }
  ++launches;

  // 2. s/2 G as three bf16 pieces; the norm pass's counters zeroed
  {
    StreamK skg{gg.p.units, gg.p.ncl, gg.p.kbtot, gg.p.maxseg};
    const int nsub = (gg.p.NC + 31) / 32;
    gram_reduce3_kernel<<<dim3(static_cast<unsigned>(gg.p.tiles), static_cast<unsigned>(nsub * nsub)), dim3(32, 8), 0,
                          cs>>>(part_g, skg, gg.p.nchunks, gg.p.NC, static_cast<int>(r), npad, static_cast<int>(rs),
                                0.5f * s, g3, cnt, ncnt);
  }
  ++launches;

  // 3. [W0 | B B B] x [A | h1 h2 h3]^T; the last epilogue warp of each quarter
  //    M tile writes n and g
  gn.p.part = part_n;
  gn.p.err = errp;
  gn.p.cnt = cnt;
  gn.p.m = m;
  gn.p.n0sq = n0sq;
  gn.p.norm = norm;
  gn.p.g = g;
  gn.p.two_s = 2.0f * s;
  gn.p.Bk = Bk;
  gn.p.ldb = static_cast<int>(ldb);
  if (launch16(gn, cs, mW0, mB, mAy_n, mG3) != cudaSuccess) {
    dora::count_launches(launches);
    return DORA_ERR_CUDA;
  }
  ++launches;
  dora::count_launches(launches);
  return dora::launch_status();
}
