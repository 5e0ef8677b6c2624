// The DoRA compose folded into the epilogue of the GEMM that produces its
// input, on GB300 (sm_103a) tensor cores.
//
// Method source: web page "人工智能训练新突破：Anthropic团队破解大模型微调内存瓶颈难题"
// (techwalker.com).  Its fused kernel merges the four elementwise passes of the
// compose into one, in the stable form
//     y = base + (g - 1) base + g s lora,
// with base = x W0^T and lora = (x A^T) B^T the products on either side.  Here
// the compose moves into the epilogue of those products, so y is written
// directly from the tensor-memory accumulator:
//
//   dora_compose_lora_fwd  (the lora up-projection):
//       acc = xa (s B)^T                       K = r, xa = x A^T (bf16)
//       y   = base + (g - 1) base + g acc      base read once, lora never stored
//   dora_linear_fwd        (both products, one K-concatenated GEMM):
//       acc = [x | xa] [W0 | s B]^T            K = in + r
//       y   = g acc                            neither base nor lora is stored
//   dora_compose_lora_fwd_bf16  (the up-projection with a bf16 B):
//       acc = xa B^T                           K = r, one product
//       y   = base + (g - 1) base + g (s acc)  s applied in the epilogue
//
// Operands are bf16, so every product is exact in fp32; the fp32 B is scaled
// by s and split into bf16 hi + lo (|lo| <= 2^-9 |hi|, residual <= 2^-17 of
// s B), and xa multiplies both (the xa segment of K is taken twice, against
// hi and against lo).  A bf16 B is taken as it is, as the linear form takes
// W0 (its first K segment), and s scales the accumulator.  Accumulation is fp32 in tensor memory; y is rounded once
// to bf16.
//
// Kernel structure (persistent, one CTA per SM, 320 threads for the linear
// form, 576 for the lora form).  On GB300 both
// forms run on CTA pairs (clusters of two CTAs on two SMs): one
// tcgen05.mma.cta_group::2 computes an M = 256 x N = 256 tile, each CTA
// holding 128 of the tokens and 128 of the weight rows, so an SM stages half
// of the weight tile.  Without cluster support the same kernel runs single
// CTAs on 128 x 256 tiles.
//   warp 0      TMA producer (each CTA its own boxes): per stage the token
//               boxes [128 x 64] and the weight boxes [128 x 64] (a pair;
//               [256 x 64] for a single CTA), 128-byte swizzle.  A pair's
//               stage is two K atoms of (x, W0) or one K atom of xa against
//               both halves of s B (xa loaded once); all copies of a stage
//               complete on the even CTA's barrier
//   warp 1      allocates 512 tensor-memory columns (two 256-column
//               accumulators, so a tile's epilogue overlaps the next tile's
//               MMAs); in the even CTA one lane issues the MMAs (8 per
//               stage) and signals both CTAs' stage-free and accumulator
//               barriers
//   warps 2..   epilogue, thread = row of the tile (its tensor-memory lane):
//               8 warps (linear form; two per tensor-memory lane quadrant,
//               two 64-column quarters of the tile each) or 16 (lora form,
//               whose epilogue is its limit; one quarter each, in two
//               32-column passes).  Each warp owns 4 KB staging
//               slots in shared memory for its 32 rows (one [32 x 64] bf16
//               box, 128-byte swizzle) and runs its own pipeline: per quarter
//               the accumulator columns, g (uniform 128-bit loads) and, for
//               the lora form, the base quarter that the warp's lane 0
//               loaded into the slot by TMA one tile ahead; y is written
//               into the slot in place and stored by TMA.  A warp frees the
//               accumulator right after its last tensor-memory load of the
//               tile, before computing y.  The epilogue warps never wait
//               for one another
// A call with an fp32 B is two launches: split_sb_kernel (s B into hi and
// lo), then this kernel as a programmatic dependent launch on it: its prologue and the
// epilogue's first base loads overlap the split, and only the producer,
// which loads hi and lo, waits for the split to complete.
// Every wait on a shared-memory barrier is bounded; a wait that gives up
// records a code in the library's device error word and all roles drain and
// leave.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace {

constexpr int kFM = 128;        // tile rows (tokens) = tensor-memory lanes
constexpr int kFN = 256;        // tile columns (outputs) = N of one MMA
constexpr int kFK = 64;         // bf16 per K block: one 128-byte swizzled row
constexpr int kFQ = 64;         // columns per epilogue quarter (one 128-byte box row)
// epilogue warps: EPI = 8 (two per tensor-memory lane quadrant, two 64-column
// quarters of a tile each) or 16 (four per quadrant, one quarter each, taken
// in two 32-column halves to bound the registers of 576 threads)
constexpr int fthreads(int epi) { return 64 + 32 * epi; }
constexpr int kGroupM = 16;     // M tiles per tile-order group of the linear form (L2 reuse of W0's tiles)
constexpr int kFMaxCtas = 256;
constexpr int kFSmemMax = 232448;
constexpr unsigned kABytes = kFM * kFK * 2;     // 16 KB
constexpr unsigned kBBytes = kFN * kFK * 2;     // 32 KB (one CTA); a CTA of a pair holds half
constexpr unsigned kSlotBytes = 32 * kFQ * 2;  // 4 KB: one warp's 32 rows of a quarter
constexpr unsigned long long kFWaitNs = 2000000000ull;

struct FusedParams {
  int T, out;
  int nseg;             // K segments: (x, W0), (xa, sB_hi), (xa, sB_lo); the lora form has the last two
  int kb[3];            // K blocks per segment
  int kbtot;            // 64-wide K blocks per tile over all segments
  int mtiles, ntiles, tiles;
  int stages;
  int na;               // token-side boxes per stage (a pair's linear form: 2)
  unsigned stage_bytes; // na token-side boxes + the weight-side boxes
  int nslots;           // staging slots per epilogue warp: one per quarter with base, else one
  int groupm;           // M tiles per tile-order group (tile_mn)
  int has_base;
  float acc_scale;      // SC kernels: the accumulator's factor in the epilogue (s)
  const float *g;
  int *err;
  const int *stall;                      // test hook: the producer withholds its loads
  const unsigned long long *limit_ns;    // limit of the bounded waits
};

// tile t's (M tile, N tile): groups of `group` M tiles, column by column
// within a group (group = 1: row by row)
__device__ __forceinline__ void tile_mn(int t, int mtiles, int ntiles, int group, int *mt, int *nt) {
  const int per = group * ntiles;
  const int grp = t / per;
  const int m0 = grp * group;
  const int gm = min(group, mtiles - m0);
  const int r = t - grp * per;
  *mt = m0 + r % gm;
  *nt = r / gm;
}

__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, uint32_t src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(src)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// this thread's bulk stores have finished reading shared memory, all but the
// most recent one (wait_read1) or all of them (wait_read0)
__device__ __forceinline__ void bulk_wait_read1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// bounded wait; the limit is read only when the phase is not yet complete
__device__ __forceinline__ bool fwait(uint32_t bar, uint32_t parity, SharedCtl *ctl, const FusedParams &p, int code) {
  if (mbar_try_wait(bar, parity)) return true;
  return wait_bounded_ns(bar, parity, ctl, p.err, code, *reinterpret_cast<const volatile unsigned long long *>(p.limit_ns));
}

// PAIR = false: one CTA per tile of 128 x 256, launched as independent CTAs.
// PAIR = true: clusters of two CTAs; a pair computes a 256 x 256 tile with
// cta_group::2 MMAs (M = 256), CTA rank c holding tokens [128 c, 128 c + 128)
// of the tile and weight rows [128 c, 128 c + 128), so each SM stages 32 KB per
// K block instead of 48.  Both CTAs' copies of a stage complete on the even
// CTA's stage barrier; the even CTA's lane issues the MMAs and signals both
// CTAs' stage-free and accumulator barriers.
// SC: the accumulator is multiplied by p.acc_scale in the epilogue (the bf16-B
// lora form, whose weight operand is B itself rather than s B)
template <bool PAIR, int EPI, bool SC = false>
__global__ void __launch_bounds__(fthreads(EPI), 1)
fused_compose_kernel(const __grid_constant__ CUtensorMap mA0, const __grid_constant__ CUtensorMap mA1,
                     const __grid_constant__ CUtensorMap mB0, const __grid_constant__ CUtensorMap mB1,
                     const __grid_constant__ CUtensorMap mB2, const __grid_constant__ CUtensorMap mC,
                     const __grid_constant__ CUtensorMap mY, const FusedParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int S = p.stages;
  static_assert(EPI == 8 || EPI == 16, "8 or 16 epilogue warps");
  constexpr int kEpiWarps = EPI;
  constexpr int kQPW = 16 / EPI;   // 64-column quarters of a tile per epilogue warp
  constexpr int kNH = EPI == 16 ? 2 : 1;   // passes per quarter
  constexpr int kCP = kFQ / kNH;           // columns per pass
  constexpr unsigned kBRows = PAIR ? kFN / 2 : kFN;   // weight rows staged by this CTA
  // weight-side boxes (64 K wide) per stage: two for a pair (8 MMAs per stage
  // wait), one for a single CTA; the token-side boxes: p.na
  constexpr int kAtoms = PAIR ? 2 : 1;
  constexpr unsigned kBAtom = kBRows * kFK * 2;
  const unsigned stage_bytes = p.stage_bytes;
  const uint32_t boff = static_cast<uint32_t>(p.na) * kABytes;   // first weight-side box of a stage
  constexpr int kTileRows = PAIR ? 2 * kFM : kFM;     // tokens per tile
  const uint32_t crank = PAIR ? cluster_ctarank() : 0u;
  const bool leader = crank == 0;
  const uint32_t peer = crank ^ 1u;
  // staging: [slot][epilogue warp][32 rows x 128 bytes]
  uint8_t *cbuf = smem + static_cast<size_t>(S) * stage_bytes;
  uint64_t *bars = reinterpret_cast<uint64_t *>(cbuf + static_cast<size_t>(p.nslots) * kEpiWarps * kSlotBytes);
  // barriers: full[S], empty[S], accf[2], acce[2], fin, cfull[2 slots][8 warps]
  SharedCtl *ctl = reinterpret_cast<SharedCtl *>(bars + 2 * S + 21);
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = full0 + 8u * S;
  const uint32_t accf0 = empty0 + 8u * S;
  const uint32_t acce0 = accf0 + 16;
  const uint32_t fin = acce0 + 16;
  const uint32_t cfull0 = fin + 8;
  const uint32_t cbase = smem_u32(cbuf);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      // a pair uses the even CTA's full barriers only
      mbar_init(full0 + 8u * s, 1);
      mbar_init(empty0 + 8u * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf0 + 8u * b, 1);
      mbar_init(acce0 + 8u * b, PAIR ? 2 * kEpiWarps : kEpiWarps);   // one arrival per epilogue warp (of both CTAs)
    }
    mbar_init(fin, 1);
    for (int k = 0; k < kQPW * kEpiWarps; ++k) mbar_init(cfull0 + 8u * k, 1);
    ctl->abort = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_map(&mA1);
    prefetch_map(&mB1);
    prefetch_map(&mB2);
    prefetch_map(&mY);
    if (p.kb[0] > 0) {
      prefetch_map(&mA0);
      prefetch_map(&mB0);
    }
    if (p.has_base) prefetch_map(&mC);
  }
  if (warp == 1) {
    __syncwarp();
    if (PAIR) {
      tmem_alloc_pair(smem_u32(&ctl->tmem_base), 512);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(&ctl->tmem_base), 512);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  // PAIR: both CTAs' barriers are initialised before either signals the other's
  if (PAIR) cluster_sync();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  // tile sequence of this CTA (of its pair: both CTAs run the same sequence)
  const int cta = static_cast<int>(PAIR ? blockIdx.x / 2 : blockIdx.x);
  const int ncta = static_cast<int>(PAIR ? gridDim.x / 2 : gridDim.x);

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------------- producer
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      // s B hi / lo come from the launch before this one (programmatic
      // dependent launch); the other roles read only the call's inputs
      pdl_wait();
      bool ok = *reinterpret_cast<const volatile int *>(p.stall) == 0;
      for (int t = cta; t < p.tiles && ok; t += ncta) {
        int mt, nt;
        tile_mn(t, p.mtiles, p.ntiles, p.groupm, &mt, &nt);
        // the tile's K blocks, segment after segment (the lora form has none in segment 0)
        for (int kb = 0; kb < p.kbtot && ok; ++kb) {
          if (!fwait(empty0 + 8u * stage, phase ^ 1u, ctl, p, 12)) {
            ok = false;
            break;
          }
          const uint32_t fb = full0 + 8u * stage;
          const uint32_t xs = smem_u32(smem + static_cast<size_t>(stage) * stage_bytes);
          int ks = kb;
          int sg = 0;
          if (ks >= p.kb[0]) {
            ks -= p.kb[0];
            sg = 1;
            if (ks >= p.kb[1]) {
              ks -= p.kb[1];
              sg = 2;
            }
          }
          const int ya = mt * kTileRows + static_cast<int>(crank) * kFM;
          const int yb = nt * kFN + static_cast<int>(crank * kBRows);
          if (PAIR) {
            // stage layout [A0][A1 (linear form)][B0][B1].  Segment 0: two K
            // atoms of x and W0.  Segment 1: one K atom of xa in A0, against
            // s B hi in B0 and s B lo in B1 (xa is loaded once for both
            // halves).  The even CTA's barrier counts both CTAs' bytes; the
            // odd CTA's copies may land before this arrival (the phase cannot
            // complete without it)
            if (leader) mbar_expect_tx(fb, 2 * (sg == 0 ? 2 * kABytes : kABytes) + 4 * kBAtom);
            const uint32_t lb = mapa_shared(fb, 0);
            if (sg == 0) {
#pragma unroll
              for (int a = 0; a < 2; ++a) {
                const int kx = (2 * ks + a) * kFK;
                tma_load_2d_pair(xs + a * kABytes, &mA0, kx, ya, lb);
                tma_load_2d_pair(xs + boff + a * kBAtom, &mB0, kx, yb, lb);
              }
            } else {
              tma_load_2d_pair(xs, &mA1, ks * kFK, ya, lb);
              tma_load_2d_pair(xs + boff, &mB1, ks * kFK, yb, lb);
              tma_load_2d_pair(xs + boff + kBAtom, &mB2, ks * kFK, yb, lb);
            }
          } else {
            mbar_expect_tx(fb, stage_bytes);
            const CUtensorMap *ma = sg == 0 ? &mA0 : &mA1;
            const CUtensorMap *mb = sg == 0 ? &mB0 : (sg == 1 ? &mB1 : &mB2);
            tma_load_2d(xs, ma, ks * kFK, ya, fb);
            tma_load_2d(xs + boff, mb, ks * kFK, yb, fb);
          }
          ++issued;
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok && issued > 0) {
        if (PAIR) {
          // the stage barriers (the even CTA's) also count the other CTA's
          // copies, which may never be issued after an abort; copies in
          // flight land within microseconds: wait 1 ms
          const unsigned long long t0 = globaltimer();
          while (globaltimer() - t0 < 1000000ull) {
          }
        } else {
          // copies in flight: the last min(issued, S) stages
          int st = stage;
          uint32_t ph = phase;
          for (int k = 0; k < S && k < issued; ++k) {
            if (--st < 0) {
              st = S - 1;
              ph ^= 1u;
            }
            wait_drain_ns(full0 + 8u * st, ph, kFWaitNs);
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ---------------------------------------------------------------- MMA issuer
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      const uint32_t idesc = PAIR ? idesc_bf16_pair(kFN) : idesc_bf16(kFN);
      // a commit arrives on the barrier of this CTA and, for a pair, on the
      // same barrier of the peer
      auto commit = [&](uint32_t bar) {
        if (PAIR) {
          mma_commit_pair(bar);
          mma_commit_pair(mapa_shared(bar, peer));
        } else {
          mma_commit(bar);
        }
      };
      int li = 0;
      for (int t = cta; t < p.tiles && ok; t += ncta, ++li) {
        const int buf = li & 1;
        const uint32_t use = static_cast<uint32_t>(li >> 1);
        if (!fwait(acce0 + 8u * buf, (use & 1u) ^ 1u, ctl, p, 13)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + static_cast<uint32_t>(buf * kFN);
        for (int kb = 0; kb < p.kbtot; ++kb) {
          if (!fwait(full0 + 8u * stage, phase, ctl, p, 14)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t xs = smem_u32(smem + static_cast<size_t>(stage) * stage_bytes);
          // a pair's segment-1 stages use A0 against both weight boxes
          const uint32_t a1 = (PAIR && kb >= p.kb[0]) ? 0u : 1u;
#pragma unroll
          for (int k = 0; k < kAtoms * kFK / 16; ++k) {
            const uint32_t a = static_cast<uint32_t>(k / (kFK / 16));             // weight box (K atom) of the stage
            const uint32_t ko = static_cast<uint32_t>(k % (kFK / 16)) * 32u;      // 16 bf16 = 32 bytes along the swizzled row
            const uint64_t ad = sdesc<32>(xs + a * a1 * kABytes + ko);
            const uint64_t bd = sdesc<32>(xs + boff + a * kBAtom + ko);
            if (PAIR) mma_bf16_ss_pair(d, ad, bd, idesc, (kb | k) != 0 ? 1u : 0u);
            else mma_bf16_ss(d, ad, bd, idesc, (kb | k) != 0 ? 1u : 0u);
          }
          commit(empty0 + 8u * stage);
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        commit(accf0 + 8u * buf);
      }
      if (PAIR) mma_commit_pair(fin);
      else mma_commit(fin);
      wait_drain_ns(fin, 0, kFWaitNs);
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    // warp e of the epilogue: tensor-memory lanes (rows of the tile) quad * 32
    // .. + 31 (a warp reaches the lane quadrant of its index mod 4), quarters
    // qb .. qb + kQPW - 1 of the tile's 256 columns
    const int e = warp - 2;
    const int quad = warp & 3;
    const int qb = (e / 4) * kQPW;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    // this warp's slot s: cbuf + (s * kEpiWarps + e) * 4 KB (1024-byte aligned,
    // so the 128-byte swizzle of a [32 x 64] box has the same phase as in a full tile)
    auto slot_off = [&](int s) { return static_cast<uint32_t>((s * kEpiWarps + e) * kSlotBytes); };
    auto cfull = [&](int s) { return cfull0 + 8u * static_cast<uint32_t>(s * kEpiWarps + e); };
    // base of this warp's quarter qb + j of tile t into slot j (lora form;
    // lane 0): the base of a tile is requested while the previous tile is
    // being written out, one tile ahead.  Per slot: whether a load was
    // issued, and the parity of the number issued (for the drain after an abort)
    uint32_t any_load = 0, load_par = 0;
    auto load_base = [&](int t, int j) {
      int mt, nt;
      tile_mn(t, p.mtiles, p.ntiles, p.groupm, &mt, &nt);
      mbar_expect_tx(cfull(j), kSlotBytes);
      tma_load_2d(cbase + slot_off(j), &mC, nt * kFN + (qb + j) * kFQ,
                  mt * kTileRows + static_cast<int>(crank) * kFM + quad * 32, cfull(j));
      any_load |= 1u << j;
      load_par ^= 1u << j;
    };
    if (p.has_base && lane == 0 && cta < p.tiles)
      for (int j = 0; j < kQPW; ++j) load_base(cta, j);
    // the staging slot of this warp's most recent TMA store (-1: none yet).
    // Before a slot is written again, every store that reads it must be done:
    // all but the most recent store when that one used another slot, else all.
    int last_slot = -1;
    int li = 0;
    bool ok = true;
    for (int t = cta; t < p.tiles && ok; t += ncta, ++li) {
      int mt, nt;
      tile_mn(t, p.mtiles, p.ntiles, p.groupm, &mt, &nt);
      const int tnext = t + ncta;
      const int buf = li & 1;
      const uint32_t use = static_cast<uint32_t>(li >> 1);
      const bool got = fwait(accf0 + 8u * buf, use & 1u, ctl, p, 15);
      if (!__all_sync(0xffffffffu, got)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int row0 = mt * kTileRows + static_cast<int>(crank) * kFM;   // this CTA's first row of the tile
      const bool rows_in = row0 + quad * 32 < p.T;   // any of this warp's rows inside y
      bool freed = false;   // this warp's arrival on the accumulator-empty barrier is done
      for (int j = 0; j < kQPW; ++j) {
        const int q = qb + j;
        const int sl = j % p.nslots;
        const int gcol0 = nt * kFN + q * kFQ;
        // a quarter entirely outside y (ragged last tiles) is neither computed
        // nor stored; warp-uniform
        const bool live = rows_in && gcol0 < p.out;
        if (p.has_base) {
          // slot j holds this tile's base quarter: the slot's load number li
          // (consumed even when the quarter is not live, to keep the phases)
          const bool gb = fwait(cfull(j), static_cast<uint32_t>(li) & 1u, ctl, p, 16);
          if (!__all_sync(0xffffffffu, gb)) {
            ok = false;
            break;
          }
        }
        if (live) {
          if (!p.has_base) {
            // the slot takes this quarter's y: earlier stores must have read it
            if (lane == 0) {
              if (last_slot == sl) bulk_wait_read0();
              else bulk_wait_read1();
            }
            __syncwarp();
          }
          uint8_t *crow = cbuf + slot_off(sl) + lane * 128;
#pragma unroll
          for (int hh = 0; hh < kNH; ++hh) {
            // g of the pass's columns: uniform 128-bit loads issued together
            // (one latency), zero past `out`
            const int c0 = gcol0 + hh * kCP;
            float4 gq[kCP / 4];
#pragma unroll
            for (int k = 0; k < kCP / 4; ++k)
              gq[k] = c0 + 4 * k < p.out ? __ldg(reinterpret_cast<const float4 *>(p.g + c0) + k)
                                         : make_float4(0.f, 0.f, 0.f, 0.f);
            float v[kCP / 32][32];
            const uint32_t col0 = static_cast<uint32_t>(buf * kFN + q * kFQ + hh * kCP);
#pragma unroll
            for (int w = 0; w < kCP / 32; ++w) tmem_ld32(lane_addr + col0 + 32 * w, v[w]);
            if (hh == kNH - 1 && j == kQPW - 1) {
              // the warp's last tensor-memory load of the tile is done: the
              // MMA lane may start the tile after next while y is computed
              tc_fence_before();
              __syncwarp();
              if (lane == 0) {
                if (PAIR) mbar_arrive_cluster(mapa_shared(acce0 + 8u * buf, 0));   // the even CTA's barrier
                else mbar_arrive(acce0 + 8u * buf);
              }
              freed = true;
            }
#pragma unroll
            for (int c = 0; c < kCP / 8; ++c) {
              // 16-byte chunk cq of the row (8 columns), at its swizzled position
              const int cq = hh * (kCP / 8) + c;
              uint4 *pc = reinterpret_cast<uint4 *>(crow + ((cq ^ (lane & 7)) << 4));
              const float *a = &v[c >> 2][(c & 3) * 8];
              const float gv[8] = {gq[2 * c].x, gq[2 * c].y, gq[2 * c].z, gq[2 * c].w,
                                   gq[2 * c + 1].x, gq[2 * c + 1].y, gq[2 * c + 1].z, gq[2 * c + 1].w};
              float yv[8];
              if (p.has_base) {
                const uint4 braw = *pc;
                const __nv_bfloat162 *bb = reinterpret_cast<const __nv_bfloat162 *>(&braw);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const float2 b2 = __bfloat1622float2(bb[e]);
                  const float a0 = SC ? p.acc_scale * a[2 * e] : a[2 * e];
                  const float a1 = SC ? p.acc_scale * a[2 * e + 1] : a[2 * e + 1];
                  yv[2 * e] = b2.x + fmaf(gv[2 * e] - 1.0f, b2.x, gv[2 * e] * a0);
                  yv[2 * e + 1] = b2.y + fmaf(gv[2 * e + 1] - 1.0f, b2.y, gv[2 * e + 1] * a1);
                }
              } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) yv[e] = gv[e] * a[e];
              }
              uint4 o;
              o.x = pack_bf16x2(yv[0], yv[1]);
              o.y = pack_bf16x2(yv[2], yv[3]);
              o.z = pack_bf16x2(yv[4], yv[5]);
              o.w = pack_bf16x2(yv[6], yv[7]);
              *pc = o;
            }
          }
          // make the writes visible to the TMA store, then lane 0 stores the
          // warp's 32 rows of the quarter
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&mY, cbase + slot_off(sl), gcol0, row0 + quad * 32);
            bulk_commit();
            last_slot = sl;
          }
        }
        if (j == kQPW - 1 && !freed) {
          // the warp's last quarter was not live, so the release after its
          // last tensor-memory load did not run: every load it made is done
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            if (PAIR) mbar_arrive_cluster(mapa_shared(acce0 + 8u * buf, 0));   // the even CTA's barrier
            else mbar_arrive(acce0 + 8u * buf);
          }
        }
        if (p.has_base && lane == 0 && j > 0 && tnext < p.tiles) {
          // slot j - 1 takes the next tile's base quarter once every store
          // that reads it is done: all but this quarter's store, if there was one
          if (live) bulk_wait_read1();
          else bulk_wait_read0();
          load_base(tnext, j - 1);
        }
      }
      if (!ok) break;
      if (p.has_base && lane == 0 && tnext < p.tiles) {
        bulk_wait_read0();
        load_base(tnext, kQPW - 1);
      }
    }
    if (lane == 0) {
      bulk_wait0();
      if (!ok) {
        // base copies that may still be in flight into this warp's slots: the
        // k-th load of a slot completes phase k - 1, of parity (count - 1) & 1
        for (int j = 0; j < kQPW; ++j)
          if ((any_load >> j) & 1u) wait_drain_ns(cfull(j), ((load_par >> j) & 1u) ^ 1u, kFWaitNs);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  // PAIR: the even CTA's MMAs (which read this CTA's shared memory and write
  // its tensor memory) are complete, and both CTAs' epilogues are done
  if (PAIR) cluster_sync();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    if (PAIR) tmem_dealloc_pair(tmem, 512);
    else tmem_dealloc(tmem, 512);
  }
}

// s B (fp32 [out, r]) -> bf16 hi = RN(s B), lo = RN(s B - hi), both [out, r]
__global__ void __launch_bounds__(256) split_sb_kernel(const float *__restrict__ B, long long n, float s,
                                                       __nv_bfloat16 *__restrict__ hi,
                                                       __nv_bfloat16 *__restrict__ lo) {
  pdl_trigger();   // the fused kernel's prologue and first base loads may start meanwhile
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const float v = s * B[i];
    const __nv_bfloat16 h = __float2bfloat16_rn(v);
    hi[i] = h;
    lo[i] = __float2bfloat16_rn(v - __bfloat162float(h));
  }
}

struct FusedPlan {
  FusedParams p;
  size_t smem_bytes;
  int ctas;
  bool pair;   // CTA pairs (fused_compose_kernel<true, .>, clusters of two)
  int epi;     // epilogue warps (the kernel instance)
};

// max_units: CTAs (one per SM) or, for pairs, the pairs that can be resident at once
// bf16_b: the lora form with a bf16 B, one K segment of r (xa, B) like the
// linear form's (x, W0)
bool plan_fused(int64_t T, int64_t in, int64_t out, int64_t r, bool has_base, bool pair, int max_units,
                FusedPlan *fp, bool bf16_b = false) {
  FusedParams &p = fp->p;
  p = FusedParams{};
  fp->pair = pair;
  // the lora form's epilogue (base read, y written per quarter) is its limit:
  // 16 warps; the linear form's MMA loop is: 8 (fewer threads and registers)
  fp->epi = has_base ? 16 : 8;
  p.T = static_cast<int>(T);
  p.out = static_cast<int>(out);
  p.nseg = bf16_b ? 1 : has_base ? 2 : 3;
  // K blocks (stages) per segment: single CTA (x, W0), (xa, s B hi), (xa, s B
  // lo), 64 K each; a pair (x, W0) by 128 K, then (xa; s B hi, s B lo) by 64 K.
  // A bf16 B: only the first segment, (xa, B) over K = r
  const int64_t k0 = bf16_b ? r : has_base ? 0 : in;
  p.kb[0] = static_cast<int>(dora::ceil_div(k0, pair ? 2 * kFK : kFK));
  p.kb[1] = bf16_b ? 0 : static_cast<int>(dora::ceil_div(r, kFK));
  p.kb[2] = pair ? 0 : p.kb[1];
  p.kbtot = p.kb[0] + p.kb[1] + p.kb[2];
  p.mtiles = static_cast<int>(dora::ceil_div(T, pair ? 2 * kFM : kFM));
  p.ntiles = static_cast<int>(dora::ceil_div(out, kFN));
  const long long tiles = static_cast<long long>(p.mtiles) * p.ntiles;
  if (tiles >= (1ll << 31)) return false;
  p.tiles = static_cast<int>(tiles);
  p.has_base = has_base ? 1 : 0;
  p.nslots = has_base ? 16 / fp->epi : 1;
  // tile order: the linear form in groups of kGroupM M tiles (W0's tiles,
  // 134 MB at the high-rank layer, are re-read from L2 across the group); the
  // lora form, whose operands stay in L2, row by row, so that concurrent
  // tiles cover whole row segments of base and y
  p.groupm = has_base ? 1 : kGroupM;
  const size_t fixed = 1024 + static_cast<size_t>(p.nslots) * fp->epi * kSlotBytes + 512;
  // a pair: two token-side boxes per stage for the linear form's (x, W0)
  // segment, one for the lora form; two half weight boxes.  A single CTA: one
  // token-side box and one weight box
  p.na = (pair && p.kb[0] > 0) ? 2 : 1;
  const size_t stage_bytes = static_cast<size_t>(p.na) * kABytes + kBBytes;
  p.stage_bytes = static_cast<unsigned>(stage_bytes);
  p.stages = static_cast<int>((kFSmemMax - fixed) / stage_bytes);
  if (p.stages > 8) p.stages = 8;
  if (p.stages < 2) return false;
  fp->smem_bytes = fixed + static_cast<size_t>(p.stages) * stage_bytes;
  const int units = p.tiles < max_units ? p.tiles : max_units;
  fp->ctas = pair ? 2 * units : units;
  return true;
}

// bf16 [rows, cols] (row stride ld elements) with a [box_rows x 64] box, 128-byte swizzle
bool map_bf16(CUtensorMap *map, const void *base, int64_t rows, int64_t cols, int64_t ld, int box_rows) {
  return make_map(map, base, true, rows, cols, ld, box_rows, 128);
}

int *g_stall_ptr[64] = {};
unsigned long long *g_limit_ptr[64] = {};
int g_max_pairs[64] = {};   // clusters of two of fused_compose_kernel<true, .> resident at once
std::atomic<int> g_pairs_allowed{1};   // test hook (dora_test_fused_pairs)

// launch configuration of the pair kernel: clusters of two CTAs along x
void pair_config(cudaLaunchConfig_t *cfg, cudaLaunchAttribute *attr, unsigned ctas, unsigned threads, size_t smem,
                 cudaStream_t cs) {
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg->gridDim = dim3(ctas);
  cfg->blockDim = dim3(threads);
  cfg->dynamicSmemBytes = smem;
  cfg->stream = cs;
  cfg->attrs = attr;
  cfg->numAttrs = 1;
}
// programmatic dependent launch on the launch before (the split of s B)
void add_pdl(cudaLaunchConfig_t *cfg, cudaLaunchAttribute *attr) {
  attr[cfg->numAttrs].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[cfg->numAttrs].val.programmaticStreamSerializationAllowed = 1;
  ++cfg->numAttrs;
}

dora_status fused_init(int device, int sms, int **errp) {
  static std::mutex mu;
  static uint64_t done_ctx[64] = {};   // context the attributes were set in
  std::lock_guard<std::mutex> lock(mu);
  if (device < 0 || device >= 64) return DORA_ERR_CUDA;
  dora_status st = dora::error_word(device, errp);
  if (st != DORA_OK) return st;
  st = dora::test_hooks(&g_stall_ptr[device], &g_limit_ptr[device]);
  if (st != DORA_OK) return st;
  const uint64_t ctx = dora::context_id();
  if (ctx == 0 || ctx != done_ctx[device]) {
    const auto a = cudaFuncAttributeMaxDynamicSharedMemorySize;
    if (cudaFuncSetAttribute(fused_compose_kernel<false, 8>, a, kFSmemMax) != cudaSuccess ||
        cudaFuncSetAttribute(fused_compose_kernel<true, 8>, a, kFSmemMax) != cudaSuccess ||
        cudaFuncSetAttribute(fused_compose_kernel<false, 16>, a, kFSmemMax) != cudaSuccess ||
        cudaFuncSetAttribute(fused_compose_kernel<true, 16>, a, kFSmemMax) != cudaSuccess ||
        cudaFuncSetAttribute(fused_compose_kernel<false, 16, true>, a, kFSmemMax) != cudaSuccess ||
        cudaFuncSetAttribute(fused_compose_kernel<true, 16, true>, a, kFSmemMax) != cudaSuccess)
      return DORA_ERR_CUDA;
    // pairs resident at once with the largest shared-memory footprint (one CTA per SM)
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    pair_config(&cfg, attr, static_cast<unsigned>(2 * (sms / 2)), fthreads(16), kFSmemMax, nullptr);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, fused_compose_kernel<true, 16>, &cfg) != cudaSuccess) {
      cudaGetLastError();
      n = 0;
    }
    g_max_pairs[device] = n;
    done_ctx[device] = dora::context_id();
  }
  return DORA_OK;
}

// shared by both entry points: x / W0 only for the linear form, base only for
// the lora form
dora_status fused_run(const void *x, const void *W0, const void *base, const void *xa, const float *B,
                      const float *g, float s, int64_t T, int64_t in, int64_t out, int64_t r, void *y,
                      void *workspace, size_t workspace_bytes, dora_stream_t stream) {
  const bool lora_form = base != nullptr;
  dora::DeviceInfo info;
  int device = 0;
  dora_status st = dora::current_device(&info, &device);
  if (st != DORA_OK) return st;
  const int sms = info.sms < kFMaxCtas ? info.sms : kFMaxCtas;
  int *errp = nullptr;
  st = fused_init(device, sms, &errp);
  if (st != DORA_OK) return st;
  // CTA pairs wherever clusters of two can be resident: each SM stages half
  // of the weight tile, the MMA lane waits once per 8 MMAs, and the lora
  // form loads xa once for both halves of s B
  const int max_pairs = g_max_pairs[device];
  const bool pair = max_pairs > 0 && g_pairs_allowed.load() != 0;
  FusedPlan fp;
  if (!plan_fused(T, in, out, r, lora_form, pair, pair ? max_pairs : sms, &fp)) return DORA_ERR_SHAPE;
  fp.p.g = g;
  fp.p.err = errp;
  fp.p.stall = g_stall_ptr[device];
  fp.p.limit_ns = g_limit_ptr[device];
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  __nv_bfloat16 *hi = static_cast<__nv_bfloat16 *>(workspace);
  __nv_bfloat16 *lo = reinterpret_cast<__nv_bfloat16 *>(static_cast<uint8_t *>(workspace) +
                                                        static_cast<size_t>(dora::round_up(out * r * 2, 256)));
  uint64_t launches = 0;
  const long long n = out * r;
  long long blocks = dora::ceil_div(n, 256);
  if (blocks > static_cast<long long>(sms) * 8) blocks = static_cast<long long>(sms) * 8;
  split_sb_kernel<<<static_cast<unsigned>(blocks), 256, 0, cs>>>(B, n, s, hi, lo);
  ++launches;

  // weight-side boxes: the whole 256-row tile, or a CTA's half of it in a pair
  const int brows = pair ? kFN / 2 : kFN;
  CUtensorMap mA0, mA1, mB0, mB1, mB2, mC, mY;
  bool ok = map_bf16(&mA1, xa, T, r, r, kFM) && map_bf16(&mB1, hi, out, r, r, brows) &&
            map_bf16(&mB2, lo, out, r, r, brows) && map_bf16(&mY, y, T, out, out, 32);
  if (lora_form) {
    ok = ok && map_bf16(&mC, base, T, out, out, 32);
    mA0 = mA1;
    mB0 = mB1;
  } else {
    ok = ok && map_bf16(&mA0, x, T, in, in, kFM) && map_bf16(&mB0, W0, out, in, in, brows);
    mC = mY;
  }
  if (!ok) {
    dora::count_launches(launches);
    return DORA_ERR_CUDA;
  }
  if (pair) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    pair_config(&cfg, attr, static_cast<unsigned>(fp.ctas), fthreads(fp.epi), fp.smem_bytes, cs);
    add_pdl(&cfg, attr);
    const cudaError_t e = fp.epi == 16
                              ? cudaLaunchKernelEx(&cfg, fused_compose_kernel<true, 16>, mA0, mA1, mB0, mB1, mB2, mC, mY,
                                                   fp.p)
                              : cudaLaunchKernelEx(&cfg, fused_compose_kernel<true, 8>, mA0, mA1, mB0, mB1, mB2, mC, mY,
                                                   fp.p);
    if (e != cudaSuccess) {
      dora::count_launches(launches);
      return DORA_ERR_CUDA;
    }
  } else {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3(static_cast<unsigned>(fp.ctas));
    cfg.blockDim = dim3(static_cast<unsigned>(fthreads(fp.epi)));
    cfg.dynamicSmemBytes = fp.smem_bytes;
    cfg.stream = cs;
    cfg.attrs = attr;
    cfg.numAttrs = 0;
    add_pdl(&cfg, attr);
    const cudaError_t e =
        fp.epi == 16
            ? cudaLaunchKernelEx(&cfg, fused_compose_kernel<false, 16>, mA0, mA1, mB0, mB1, mB2, mC, mY, fp.p)
            : cudaLaunchKernelEx(&cfg, fused_compose_kernel<false, 8>, mA0, mA1, mB0, mB1, mB2, mC, mY, fp.p);
    if (e != cudaSuccess) {
      dora::count_launches(launches);
      return DORA_ERR_CUDA;
    }
  }
  ++launches;
  dora::count_launches(launches);
  return dora::launch_status();
}

// the lora form with a bf16 B: one launch, no split (B is the MMA operand as
// it is; s scales the accumulator)
dora_status fused_run_bf16b(const void *base, const void *xa, const void *B, const float *g, float s, int64_t T,
                            int64_t out, int64_t r, void *y, dora_stream_t stream) {
  dora::DeviceInfo info;
  int device = 0;
  dora_status st = dora::current_device(&info, &device);
  if (st != DORA_OK) return st;
  const int sms = info.sms < kFMaxCtas ? info.sms : kFMaxCtas;
  int *errp = nullptr;
  st = fused_init(device, sms, &errp);
  if (st != DORA_OK) return st;
  const int max_pairs = g_max_pairs[device];
  const bool pair = max_pairs > 0 && g_pairs_allowed.load() != 0;
  FusedPlan fp;
  if (!plan_fused(T, 0, out, r, true, pair, pair ? max_pairs : sms, &fp, true)) return DORA_ERR_SHAPE;
  fp.p.g = g;
  fp.p.acc_scale = s;
  fp.p.err = errp;
  fp.p.stall = g_stall_ptr[device];
  fp.p.limit_ns = g_limit_ptr[device];
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  uint64_t launches = 0;
  const int brows = pair ? kFN / 2 : kFN;
  CUtensorMap mA0, mB0, mC, mY;
  const bool ok = map_bf16(&mA0, xa, T, r, r, kFM) && map_bf16(&mB0, B, out, r, r, brows) &&
                  map_bf16(&mC, base, T, out, out, 32) && map_bf16(&mY, y, T, out, out, 32);
  if (!ok) return DORA_ERR_CUDA;
  // an ordinary launch: the epilogue reads base from the first instruction, so
  // the kernel may not start before the launch that wrote it has completed
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cudaError_t e;
  if (pair) {
    pair_config(&cfg, attr, static_cast<unsigned>(fp.ctas), fthreads(16), fp.smem_bytes, cs);
    e = cudaLaunchKernelEx(&cfg, fused_compose_kernel<true, 16, true>, mA0, mA0, mB0, mB0, mB0, mC, mY, fp.p);
  } else {
    cfg.gridDim = dim3(static_cast<unsigned>(fp.ctas));
    cfg.blockDim = dim3(static_cast<unsigned>(fthreads(16)));
    cfg.dynamicSmemBytes = fp.smem_bytes;
    cfg.stream = cs;
    cfg.attrs = attr;
    cfg.numAttrs = 0;
    e = cudaLaunchKernelEx(&cfg, fused_compose_kernel<false, 16, true>, mA0, mA0, mB0, mB0, mB0, mC, mY, fp.p);
  }
  if (e != cudaSuccess) return DORA_ERR_CUDA;
  ++launches;
  dora::count_launches(launches);
  return dora::launch_status();
}

}  // namespace

extern "C" size_t dora_compose_fused_workspace(int64_t out, int64_t r) {
  if (out < 0 || r < 1 || out >= (1ll << 31) || r >= (1ll << 20)) return 0;
  const size_t piece = static_cast<size_t>(dora::round_up(out * r * 2, 256));
  return piece > 0 ? 2 * piece : 256;
}

namespace {
dora_status fused_check(const void *xa, const float *B, const float *g, int64_t T, int64_t out, int64_t r, void *y,
                        void *workspace, size_t workspace_bytes) {
  if (!xa || !B || !g || !y) return DORA_ERR_NULL;
  if (!workspace) return DORA_ERR_WORKSPACE;
  // TMA: 16-byte aligned bases and row strides (bf16 rows of out and r elements)
  if (out % 8 != 0 || r % 8 != 0) return DORA_ERR_ALIGN;
  if (!dora::aligned(xa, 16) || !dora::aligned(y, 16) || !dora::aligned(B, 4) || !dora::aligned(g, 16))
    return DORA_ERR_ALIGN;
  if (!dora::aligned(workspace, 256) || workspace_bytes < dora_compose_fused_workspace(out, r))
    return DORA_ERR_WORKSPACE;
  (void)T;
  return DORA_OK;
}
}  // namespace

extern "C" dora_status dora_compose_lora_fwd(const void *base, const void *xa, const float *B, const float *g, float s,
                                             int64_t T, int64_t out, int64_t r, void *y, void *workspace,
                                             size_t workspace_bytes, dora_stream_t stream) {
  if (T < 0 || out < 0 || r < 1 || T >= (1ll << 31) || out >= (1ll << 31) || r >= (1ll << 20)) return DORA_ERR_SHAPE;
  if (T == 0 || out == 0) return DORA_OK;
  if (!base) return DORA_ERR_NULL;
  dora_status st = fused_check(xa, B, g, T, out, r, y, workspace, workspace_bytes);
  if (st != DORA_OK) return st;
  if (!dora::aligned(base, 16)) return DORA_ERR_ALIGN;
  return fused_run(nullptr, nullptr, base, xa, B, g, s, T, 0, out, r, y, workspace, workspace_bytes, stream);
}

extern "C" dora_status dora_linear_fwd(const void *x, const void *W0, const void *xa, const float *B, const float *g,
                                       float s, int64_t T, int64_t in, int64_t out, int64_t r, void *y,
                                       void *workspace, size_t workspace_bytes, dora_stream_t stream) {
  if (T < 0 || out < 0 || in < 1 || r < 1 || T >= (1ll << 31) || out >= (1ll << 31) || in >= (1ll << 31) ||
      r >= (1ll << 20))
    return DORA_ERR_SHAPE;
  if (T == 0 || out == 0) return DORA_OK;
  if (!x || !W0) return DORA_ERR_NULL;
  dora_status st = fused_check(xa, B, g, T, out, r, y, workspace, workspace_bytes);
  if (st != DORA_OK) return st;
  if (in % 8 != 0 || !dora::aligned(x, 16) || !dora::aligned(W0, 16)) return DORA_ERR_ALIGN;
  return fused_run(x, W0, nullptr, xa, B, g, s, T, in, out, r, y, workspace, workspace_bytes, stream);
}

extern "C" dora_status dora_compose_lora_fwd_bf16(const void *base, const void *xa, const void *B, const float *g,
                                                  float s, int64_t T, int64_t out, int64_t r, void *y,
                                                  dora_stream_t stream) {
  if (T < 0 || out < 0 || r < 1 || T >= (1ll << 31) || out >= (1ll << 31) || r >= (1ll << 20)) return DORA_ERR_SHAPE;
  if (T == 0 || out == 0) return DORA_OK;
  if (!base || !xa || !B || !g || !y) return DORA_ERR_NULL;
  // TMA: 16-byte aligned bases and row strides (bf16 rows of out and r elements)
  if (out % 8 != 0 || r % 8 != 0) return DORA_ERR_ALIGN;
  if (!dora::aligned(base, 16) || !dora::aligned(xa, 16) || !dora::aligned(B, 16) || !dora::aligned(y, 16) ||
      !dora::aligned(g, 16))
    return DORA_ERR_ALIGN;
  return fused_run_bf16b(base, xa, B, g, s, T, out, r, y, stream);
}

extern "C" dora_status dora_test_fused_pairs(int allow) {
  g_pairs_allowed.store(allow ? 1 : 0);
  return DORA_OK;
}
