// attn_kernel.cuh -- head-major non-causal attention forward for sm_103a.
//
// Computes, per (batch*head) bh and query row i,
//     out[bh, i, :] = sum_j softmax_j(q[bh,i,:] . k[bh,j,:]) v[bh, j, :]
// as in the WGSL shader "vision_attention_flash_sub_hpd_f16.wgsl"
// (rullama 0.1.0): q/k/v rounded to f16, scores and P.V accumulated in f32,
// f32 online softmax with running (m, l, o), no 1/sqrt(head_dim) factor.
//
// Operands (input mode kIn; every mode rounds f32 to f16 to nearest even,
// as the staging kernel does, so all give bit-identical results):
//   kInF16     the f16 copies written by vattn_stage_kernel
//              (stage_kernel.cuh), [B*H, N, d_pad] f16, d_pad = head_dim
//              rounded up to 16, zero padding, by TMA;
//   kInF32     (two query tiles, head_dim <= 64) the caller's f32 tensors:
//              TMA brings f32 tiles into a ring of shared-memory slots and a
//              fourth warpgroup rounds them into the swizzled operand tiles;
//   kInF32Q    k, v as kInF16; q in f32, rounded by warp 3 once per work
//              tile;
//   kInStageKV q as kInF32Q; a fourth warpgroup writes the f16 copies of k
//              and v itself (each key tile once, by one block of the
//              cooperative grid, which then sets the tile's ready flag), and
//              the K/V producer of every block waits for a tile's flag
//              before reading it by TMA as in kInF16.
// The shader's design (8 queries x 32 keys per 64-thread workgroup, scalar
// dot products, subgroup reductions) is replaced by a GB300 one:
//   * a work tile = one bh and NQ query tiles of 128 rows; the grid is one
//     block per multiprocessor and each block loops over its tiles, so
//     barrier setup and TMEM allocation happen once, and the next tile's
//     K/V and Q loads and first S = Q K^T overlap the end of the current one;
//   * warp 0 streams the f16 K and V tiles, warp 3 the Q tiles, with TMA
//     (cp.async.bulk.tensor, 128-byte swizzle) straight into the layout the
//     tensor core reads; rows past n_patches read as zero;
//   * warp 1 issues the tcgen05.mma of S = Q K^T (f32 in TMEM), warp 2
//     those of O += P V (P from TMEM, V from shared memory).  Each waits at
//     one point per key tile, so one keeps the tensor core busy while the
//     other waits or is held back by the softmax warps on its scheduler.
//     S and P have separate TMEM columns: the next S = Q K^T is issued as
//     soon as the softmax has copied the current S into registers, and the
//     softmax computes its exponentials while the previous P V still runs;
//   * one warpgroup per query tile runs the online softmax: thread = query
//     row, so the row max and row sum need no shuffles; exp is exp2 with
//     log2(e) folded into one FMA; O is rescaled in TMEM only when the
//     row max grew by more than 2^8 (exact after the final 1/l);
//   * the same warpgroup divides by l and stores its rows of out (f32);
//   * the producers wait for the previous kernel (griddepcontrol.wait)
//     before their first load, so with a programmatic launch the block
//     prologue overlaps the end of the staging pass;
//   * 384 threads (control warpgroup + two softmax warpgroups), or 512 with
//     the fourth warpgroup of kInF32 / kInStageKV; setmaxnreg gives the
//     softmax warps 224 (216 with 512 threads) registers and the others 56
//     (40).
// TMEM columns (512): S buffers [0,128) and [128,256); with two query tiles
// P0, P1 at 256, 320 and O0, O1 at 384, 448 (head_dim <= 64), or one P
// buffer at 256 that the two tiles take in turn, half (64 keys) by half,
// and O0, O1 at 320, 416 (head_dim 65..96); with one query tile P at 256
// and O at 320 (head_dim <= 128; the accurate mode: P hi 256, P lo 320, O
// 384).
// Every wait is bounded: on timeout the block records the wait site in
// g_vattn_status, raises a shared abort flag so the other roles leave their
// loops, drains its own TMA copies and MMAs, frees TMEM and exits.
#pragma once

#include <cuda.h>
#include <cstdint>

#include "ptx.cuh"

namespace vattn {

constexpr int kBM = 128;  // query rows per tile (UMMA M)
constexpr int kBN = 128;  // keys per K/V tile (UMMA N of S, K of P.V)
constexpr int kBoxBytes = 128 * 128;  // one TMA box: 128 rows x 64 f16
constexpr uint32_t kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleLog2 = 8.0f;                 // lazy-rescale threshold
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;   // 2 s per wait

// g_vattn_status: bit 8 = a wait timed out; low byte = the wait site.
enum WaitSite : uint32_t {
  kSiteProducerK = 1,
  kSiteProducerV = 2,
  kSiteProducerQ = 3,
  kSiteMmaQ = 5,
  kSiteMmaK = 6,
  kSiteMmaV = 7,
  kSiteMmaP = 8,
  kSiteSoftS = 9,
  kSiteSoftO = 10,
  kSiteEpilogue = 11,
  kSiteDrainTma = 12,
  kSiteDrainMma = 13,
  kSiteMmaSFree = 14,
  kSiteConvert = 16,
  kSiteKvReady = 17,
  kSitePartial = 18,
};
constexpr uint32_t kStatusTimeout = 0x100u;

__device__ uint32_t g_vattn_status;

struct Params {
  float* out;       // f32 output (kOut16 == false)
  uint16_t* out16;  // f16 output (kOut16 == true): IEEE binary16, round to nearest even
  int n_patches;  // N
  int head_dim;   // D
  int d_pad;      // D rounded up to 16
  int n_qblocks;  // query blocks (NQ tiles of 128 rows) per bh
  int n_tiles;    // bh * n_qblocks units of work, spread over the grid
  int n_ktiles;   // ceil(N / kBN)
  int vec_out;    // out rows may be written with 16-byte stores
  int tma_out;    // write out through tm_o (TMA stores; head_dim <= 64, % 4 == 0)
  // kInStageKV only: the f16 copies [B*H, N, d_pad] of k and v that the
  // kernel writes (from the f32 maps tm_kl / tm_vl) and tm_k / tm_v read,
  // and one ready flag per (bh, key tile), zero at launch
  uint16_t* k16;
  uint16_t* v16;
  uint32_t* kv_ready;
  // Work schedule (see Sched): `rounds` rounds of whole tiles, one more
  // whole tile for the first `extra` blocks, then the remaining tiles' key
  // tiles (tail_units of them) cut into one contiguous range per block.  A
  // tile cut between blocks b and b + 1 is finished by whichever of its two
  // parts ends second: the first one leaves its partial (O, m, l) in
  // part[slot b] and raises its flag in part_sync, the second merges.
  int rounds;
  int extra;
  long long tail_units;
  float* part;          // [n_blocks - 1][NQ][128 rows x (d_pad + 2)] f32, or null
  uint32_t* part_sync;  // [n_blocks - 1][NQ][4 warps][2]: arrival count, ready flag; zero at launch
};

// A block's share of the work, in order: whole tiles blockIdx.x + r *
// gridDim.x for r < rounds, whole tile blockIdx.x + rounds * gridDim.x if
// blockIdx.x < extra, then the key-tile units [u0, u1) of its range of the
// tail (tiles (rounds + (extra > 0)) * gridDim.x onwards, unit u = key tile
// u % T of tail tile u / T).  A schedule has either whole extra tiles or a
// tail.  Every range of the tail holds at least T units (the host chooses
// `rounds` so), so a tile is cut at most once, between two neighbouring
// blocks.
struct Piece {
  int tile;  // bh * n_qblocks + query block
  int j0;    // key tiles [j0, j1)
  int j1;
  int slot;  // partial slot of a cut tile (-1: a whole tile)
};

// The block's schedule, computed once by thread 0 into shared memory (so
// that no role keeps it in registers) and read back per piece.
struct Sched {
  int whole;      // whole tiles of this block: rounds (+ 1 if blockIdx.x < extra)
  int tail_base;  // first tile of the tail
  int x0, jf;     // the first tail piece: tail tile x0 from key tile jf
  int x1, jl;     // the last tail piece: tail tile x1 up to key tile jl (exclusive)
  int n;          // pieces of this block

  __device__ __forceinline__ static Sched make(const Params& p, int T) {
    Sched s;
    const int G = static_cast<int>(gridDim.x);
    const int b = static_cast<int>(blockIdx.x);
    s.whole = p.rounds + (b < p.extra ? 1 : 0);
    s.tail_base = p.rounds * G;
    const long long u0 = static_cast<long long>(b) * p.tail_units / G;
    const long long u1 = static_cast<long long>(b + 1) * p.tail_units / G;
    s.x0 = static_cast<int>(u0 / T);
    s.jf = static_cast<int>(u0 - static_cast<long long>(s.x0) * T);
    s.x1 = u1 > u0 ? static_cast<int>((u1 - 1) / T) : s.x0 - 1;
    s.jl = u1 > u0 ? static_cast<int>(u1 - static_cast<long long>(s.x1) * T) : 0;
    s.n = s.whole + (s.x1 - s.x0 + 1);
    return s;
  }
};

// Piece i of the block whose Sched sits in shared memory at `sp`.
__device__ __forceinline__ Piece piece_at(const volatile Sched* sp, int i, int T) {
  const int b = static_cast<int>(blockIdx.x);
  if (i < sp->whole) return Piece{b + i * static_cast<int>(gridDim.x), 0, T, -1};
  const int x0 = sp->x0;
  const int x = x0 + (i - sp->whole);
  Piece pc;
  pc.tile = sp->tail_base + x;
  pc.j0 = x == x0 ? sp->jf : 0;
  pc.j1 = x == sp->x1 ? sp->jl : T;
  pc.slot = pc.j0 > 0 ? b - 1 : (pc.j1 < T ? b : -1);
  return pc;
}

// Shared-memory plan for NQ query tiles and NKB 64-column blocks of d_pad.
// f16 tiles: NKB blocks of [128 rows x 128 bytes], 128-byte swizzle.
// kAcc (accurate mode, one query tile): every Q, K and V tile comes as an
// f16 pair (hi, lo), the lo part right after the hi part.
// kIn (two query tiles, head_dim <= 64 for kInF32 and kInF32Q): where the
// operands come from.
//   kInF16:  q, k, v f16 copies (the staging kernel's), TMA into the tiles;
//   kInF32:  q, k, v f32 tiles [128 rows x 64 columns] into a ring of two
//            slots; a fourth warpgroup rounds them to f16 into the same
//            swizzled tiles (three K/V stages);
//   kInF32Q: k, v f16 copies; q f32 tiles into two slots (one per query
//            tile), rounded to f16 by warp 3 once per work tile;
//   kInStageKV: as kInF32Q, and a fourth warpgroup writes the f16 copies of
//            k and v itself (global to global, each key tile once, ahead of
//            the blocks that read it, which wait for its ready flag).
constexpr int kInF16 = 0, kInF32 = 1, kInF32Q = 2, kInStageKV = 3;

template <int NQ, int NKB, bool kAcc = false, int kIn = kInF16>
struct Plan {
  static constexpr bool kF32 = kIn == kInF32;                         // every operand from f32
  static constexpr bool kStageKV = kIn == kInStageKV;                 // k, v copies written here
  static constexpr bool kF32Q = kIn == kInF32Q || kIn == kInStageKV;  // q from f32
  static constexpr bool kConvWG = kF32 || kStageKV;                   // a fourth warpgroup
  // control warpgroup + one softmax warpgroup per query tile (+ converters)
  static constexpr int kThreads = 128 * (1 + NQ) + (kConvWG ? 128 : 0);
  static constexpr int kTileF16 = NKB * kBoxBytes;
  static constexpr int kParts = kAcc ? 2 : 1;      // f16 terms per operand
  static constexpr int kPartBytes = kTileF16;      // offset of lo after hi
  static constexpr int kStageStride = kParts * kTileF16;
  static constexpr int kStages =  // K and V stages
      kF32 ? 3 : (kStageKV ? 2 : (kF32Q ? 3 : (kAcc ? (NKB == 1 ? 3 : 1) : (NKB == 1 ? 5 : (NQ == 2 ? 2 : 3)))));
  // two query tiles with head_dim > 64: O needs 2 x 80..128 TMEM columns, so
  // the two tiles take turns with one P buffer
  static constexpr bool kSharedP = NQ == 2 && NKB == 2;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + NQ * kStageStride;
  static constexpr int kOffV = kOffK + kStages * kStageStride;
  // output staging for the TMA-store epilogue (head_dim <= 64 only): two
  // 2 KB buffers (32 rows x 16 f32, 64-byte swizzle) per softmax warp
  static constexpr int kEpiBytes = (NKB == 1 && !kAcc) ? 4 * NQ * 4096 : 0;
  static constexpr int kOffEpi = kOffV + kStages * kStageStride;
  // f32 slots: the kInF32 ring; one per query tile for kInF32Q; and for
  // kInStageKV one more, slot NQ, for the k / v tiles being staged
  static constexpr int kF32Slots = kF32 ? 2 : (kStageKV ? NQ + 1 : (kF32Q ? NQ : 0));
  static constexpr int kF32TileBytes = kBM * 64 * 4;  // 128 rows x 64 f32, unswizzled
  static constexpr int kOffF32 = kOffEpi + kEpiBytes;
  static constexpr int kOffBar = kOffF32 + kF32Slots * kF32TileBytes;
  static constexpr int kBarBytes = 512;
  static constexpr int kSmemBytes = kOffBar + kBarBytes + 1024;  // + alignment slack
  // register split (two query tiles): control warpgroup 56, softmax 224;
  // launch gives 65536 / 384 -> 168 per thread, 56 + 2 * 224 <= 3 * 168.
  // With the converter warpgroup: 65536 / 512 -> 128 per thread,
  // 2 * 40 + 2 * 216 <= 4 * 128.
  static constexpr bool kSplitRegs = NQ == 2;
  static constexpr uint32_t kRegsSoftmax = kConvWG ? 216 : 224;
  static constexpr uint32_t kRegsOther = kConvWG ? 40 : 56;
  static constexpr uint32_t kRegsLaunch = kConvWG ? 128 : 168;
  // TMEM columns: S buffers at 0 and 128, P at 256 (kAcc: P lo at 320), O
  // after them; two query tiles keep their P (and O) blocks kColPStride
  // (kColOStride) apart.  Shared P (two query tiles, head_dim > 64): one P
  // block at 256 and O blocks at 320 and 416, so d_pad <= 96.
  static constexpr uint32_t kColP = 256;
  static constexpr uint32_t kColPlo = 320;
  static constexpr uint32_t kColO = kSharedP ? 320 : ((NQ == 2 || kAcc) ? 384 : 320);
  static constexpr uint32_t kColPStride = kSharedP ? 0 : 64;
  static constexpr uint32_t kColOStride = kSharedP ? 96 : 64;
  static_assert(!kSplitRegs || (kConvWG ? 2 : 1) * kRegsOther + NQ * kRegsSoftmax <=
                                    static_cast<uint32_t>(kThreads / 128) * kRegsLaunch,
                "register split too large");
  static_assert(kIn == kInF16 || (NQ == 2 && NKB == 1 && !kAcc),
                "f32 inputs: two query tiles, head_dim <= 64");
  static_assert(kF32Slots <= 4, "f32 ring barriers");
  static_assert(kSmemBytes <= 232448, "shared memory plan exceeds 227 KB");
  static_assert(!kSharedP || !kAcc, "shared P is for the f16 path");
  static_assert(!kAcc || NQ == 1, "the accurate mode takes one query tile");
};

// mbarrier indices inside the barrier block (kStages <= 5).
enum Bar : int {
  kBarQFull = 0,      // Q tiles landed                     (1 + tx; f32 inputs: 4 per tile)
  kBarKFull = 1,      // [5] K stage landed                 (1 + tx; f32 inputs: 4)
  kBarKEmpty = 6,     // [5] S MMAs done with K stage       (commit)
  kBarVFull = 11,     // [5] V stage landed                 (1 + tx; f32 inputs: 4)
  kBarVEmpty = 16,    // [5] P.V MMAs done with V stage     (commit)
  kBarSFull = 21,     // [2] S buffer complete in TMEM      (commit)
  kBarSFree = 23,     // [2] S buffer(s) copied to registers (one per softmax warp;
                      //     two query tiles share barrier 0)
  kBarPFull = 25,     // P of every query tile written, O rescaled (one per softmax warp)
  kBarODone = 27,     // [2] P.V of query tile complete     (commit)
  kBarMmaDone = 29,   // every MMA of the block complete    (one commit per issuer)
  kBarQEmpty = 30,    // S products of a tile done with its Q tiles (commit)
  kBarF32Full = 31,   // [4] f32 ring slot landed           (1 + tx)
  kBarF32Empty = 35,  // [4] f32 ring slot read (one per converter warp)
  kBarQFull1 = 39,    // kInF32Q: Q tile 1 rounded (Q tile 0: kBarQFull)
  kBarPHalf = 40,     // [2] shared P: first half (keys 0..63) of P written (one per softmax warp)
  kBarOHalf = 42,     // [2] shared P: P.V of the first half complete (commit)
  kNumBars = 44,
};
constexpr int kTmemSlotOff = kNumBars * 8;   // u32 TMEM base address
constexpr int kAbortOff = kTmemSlotOff + 4;  // u32 abort flag
constexpr int kConvOkOff = kAbortOff + 4;    // u32: kInStageKV slot wait result, for the warpgroup
constexpr int kSchedOff = kConvOkOff + 4;    // Sched of the block
static_assert(kSchedOff + sizeof(Sched) <= 512, "barrier block overflow");

struct Waiter {
  volatile uint32_t* abort_flag;

  // Bounded wait that also gives up when another role has aborted.
  __device__ __forceinline__ bool wait(uint32_t bar, uint32_t parity, uint32_t site) const {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::global_timer_ns();
    for (uint32_t it = 1;; ++it) {
      if (ptx::mbar_try_wait(bar, parity)) return true;
      if ((it & 31u) == 0) {
        if (*abort_flag) return false;
        if (ptx::global_timer_ns() - t0 > kWaitTimeoutNs) {
          *abort_flag = 1;
          atomicOr(&g_vattn_status, kStatusTimeout | site);
          return false;
        }
      }
    }
  }

  // Bounded wait for a flag in global memory that another block sets
  // (release) once what it guards is written; acquire on success.
  __device__ __forceinline__ bool wait_flag(const uint32_t* f, uint32_t site) const {
    if (ptx::ld_acquire_gpu(f) != 0) return true;
    const uint64_t t0 = ptx::global_timer_ns();
    for (uint32_t it = 1;; ++it) {
      __nanosleep(64);
      if (ptx::ld_acquire_gpu(f) != 0) return true;
      if ((it & 15u) == 0) {
        if (*abort_flag) return false;
        if (ptx::global_timer_ns() - t0 > kWaitTimeoutNs) {
          *abort_flag = 1;
          atomicOr(&g_vattn_status, kStatusTimeout | site);
          return false;
        }
      }
    }
  }

  // Warp-uniform variant: all lanes leave together.
  __device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, uint32_t site) const {
    const bool ok = wait(bar, parity, site);
    return __all_sync(0xffffffffu, ok);
  }

  // Bounded wait that ignores the abort flag: used while draining copies
  // and MMAs before the block exits.
  __device__ __forceinline__ bool drain(uint32_t bar, uint32_t parity, uint32_t site) const {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::global_timer_ns();
    for (uint32_t it = 1;; ++it) {
      if (ptx::mbar_try_wait(bar, parity)) return true;
      if ((it & 31u) == 0 && ptx::global_timer_ns() - t0 > kWaitTimeoutNs) {
        atomicOr(&g_vattn_status, kStatusTimeout | site);
        return false;
      }
    }
  }
};

// One arrival per warp: the lanes' earlier memory operations are ordered
// before lane 0's (release) arrive by the warp barrier.
__device__ __forceinline__ void warp_arrive(uint32_t bar) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) ptx::mbar_arrive(bar);
}

// Persistent: tile = bh * n_qblocks + query block, n_tiles in all; block b
// handles tiles b, b + gridDim.x, ... (gridDim.x <= n_tiles).
// tm_q / tm_k / tm_v: f16 [B*H, N, d_pad] with boxes of {64 columns, 128 rows},
// 128-byte swizzle (columns past d_pad and rows past N read as zero).
// kOut16: the output is rounded to f16 (round to nearest even) instead of
// written in f32.
// kAcc: accurate mode.  q, k, v arrive as f16 pairs (hi, lo; the lo tensor
// maps are tm_ql, tm_kl, tm_vl), the softmax weights are split the same way
// into P hi and P lo, and each product takes three MMAs:
//   S = Qh Kh^T + Qh Kl^T + Ql Kh^T,   O += Ph Vh + Ph Vl + Pl Vh
// (the lo x lo terms are below 2^-22 relative).
// kIn == kInF32: tm_q / tm_k / tm_v are f32 [B*H, N, head_dim] maps with
// boxes of {64 columns, 128 rows}, no swizzle (head_dim % 4 == 0, <= 64);
// warp 0 streams the tiles (per work tile: K_0, V_0, Q_0, Q_1, K_1, V_1, ...)
// into the f32 ring, and warps 12..15 round each one to f16 into its swizzled
// Q, K or V tile (the f16 staging pass is not needed).
// kIn == kInF32Q: tm_q is such an f32 map and tm_k / tm_v the f16 ones; warp
// 3 loads the next work tile's Q tiles into their f32 slots while the
// current one runs and rounds them into the Q tiles once the S products are
// done with the old ones (the staging pass then only rounds k and v).
template <int NQ, int NKB, bool kOut16 = false, bool kAcc = false, int kIn = kInF16>
__global__ void __launch_bounds__(Plan<NQ, NKB, kAcc, kIn>::kThreads, 1)
    vattn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v,
                     const __grid_constant__ CUtensorMap tm_o,
                     const __grid_constant__ CUtensorMap tm_ql,
                     const __grid_constant__ CUtensorMap tm_kl,
                     const __grid_constant__ CUtensorMap tm_vl, const Params p) {
  using P = Plan<NQ, NKB, kAcc, kIn>;
  constexpr bool kF32 = P::kF32;
  constexpr int kRing = P::kF32Slots > 0 ? P::kF32Slots : 1;  // f32 ring size (index arithmetic)
  constexpr int S = P::kStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_s = ptx::smem_addr(smem_raw);
  const uint32_t base_s = (raw_s + 1023u) & ~1023u;
  uint8_t* const base = smem_raw + (base_s - raw_s);
  const uint32_t bar0 = base_s + P::kOffBar;
  auto bar = [bar0](int i) -> uint32_t { return bar0 + 8u * static_cast<uint32_t>(i); };
  volatile uint32_t* abort_flag =
      reinterpret_cast<volatile uint32_t*>(base + P::kOffBar + kAbortOff);
  const Waiter w{abort_flag};

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int N = p.n_patches;
  const int T = p.n_ktiles;
  // The pieces of work of this block (Sched, in shared memory once the
  // block's first barrier has passed); every block has at least one.
  const volatile Sched* sched_s = reinterpret_cast<const volatile Sched*>(base + P::kOffBar + kSchedOff);
  auto sched = [&](int i) -> Piece { return piece_at(sched_s, i, T); };
  auto tile_bh = [&](int i) -> int { return sched(i).tile / p.n_qblocks; };
  auto tile_row0 = [&](int i) -> int { return (sched(i).tile % p.n_qblocks) * (kBM * NQ); };

  // Key tiles are numbered across the tiles of the block (g = i * T + j), so
  // every ring of barriers keeps its phase from one tile to the next.
  // S buffer of query tile t for key tile g, and the phase of its barriers
  auto sbuf = [](int t, int64_t g) -> int { return NQ == 2 ? t : static_cast<int>(g & 1); };
  auto sphase = [](int64_t g) -> uint32_t {
    return NQ == 2 ? static_cast<uint32_t>(g & 1) : static_cast<uint32_t>((g >> 1) & 1);
  };
  // barrier telling that the S buffer of key tile g was copied to registers
  auto sfree_bar = [](int64_t g) -> int { return NQ == 2 ? 0 : static_cast<int>(g & 1); };
  // K/V stage of key tile g and the phase of its barriers
  auto kv_stage = [](int64_t g) -> int { return static_cast<int>(g % S); };
  auto kv_phase = [](int64_t g) -> uint32_t { return static_cast<uint32_t>((g / S) & 1); };

  if (threadIdx.x == 0) {
    // f32 inputs: the converter warps (four) arrive on the f16 tiles' barriers
    ptx::mbar_init(bar(kBarQFull), kF32 ? 4 * NQ : 1);  // kInF32Q: warp 3, Q tile 0
    ptx::mbar_init(bar(kBarQFull1), 1);                 // kInF32Q: warp 3, Q tile 1
    ptx::mbar_init(bar(kBarQEmpty), 1);
    for (int i = 0; i < S; ++i) {
      ptx::mbar_init(bar(kBarKFull + i), kF32 ? 4 : 1);
      ptx::mbar_init(bar(kBarKEmpty + i), 1);
      ptx::mbar_init(bar(kBarVFull + i), kF32 ? 4 : 1);
      ptx::mbar_init(bar(kBarVEmpty + i), 1);
    }
    for (int i = 0; i < P::kF32Slots; ++i) {
      ptx::mbar_init(bar(kBarF32Full + i), 1);
      ptx::mbar_init(bar(kBarF32Empty + i), 4);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(bar(kBarSFull + i), 1);
      ptx::mbar_init(bar(kBarSFree + i), NQ == 2 ? 8 : 4);
      ptx::mbar_init(bar(kBarPFull + i), P::kSharedP ? 4 : 4 * NQ);
      ptx::mbar_init(bar(kBarODone + i), 1);
      ptx::mbar_init(bar(kBarPHalf + i), 4);
      ptx::mbar_init(bar(kBarOHalf + i), 1);
    }
    ptx::mbar_init(bar(kBarMmaDone), 2);
    *abort_flag = 0;
    *reinterpret_cast<Sched*>(base + P::kOffBar + kSchedOff) = Sched::make(p, T);
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(bar0 + kTmemSlotOff, kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(base + P::kOffBar + kTmemSlotOff);
  const int n_mine = sched_s->n;
  const uint32_t tile_bytes = static_cast<uint32_t>(P::kTileF16);

  const bool softmax_wg = warp >= 4 && warp < 4 + 4 * NQ;
  const bool convert_wg = P::kConvWG && warp >= 4 + 4 * NQ;
  if (P::kStageKV && convert_wg) {
    if (P::kSplitRegs) ptx::regs_decrease<P::kRegsOther>();
    // ------------------------------------------- k, v staging, in the kernel
    // Job s = one key tile (bh, j) of k and v: its rows come by TMA as f32
    // [128 x 64] into f32 slot NQ (tm_kl / tm_vl: f32 maps, columns past
    // head_dim and rows past N read as zero), are rounded to f16 rows of d_pad
    // columns into the copies that tm_k / tm_v read (rows < N only), and
    // kv_ready[bh * T + j] is set (release).  Block b takes jobs b,
    // b + gridDim.x, ... of a sequence ordered by when they are needed: the
    // heads whose first work tile falls in round r (work tiles r * gridDim.x
    // .. (r + 1) * gridDim.x - 1) come before those of round r + 1, and
    // within a round key tile j of all of them before key tile j + 1.
    // Thread c of the 128 handles 8-column chunks c, c + 128, ... of a tile.
    const int tid = static_cast<int>(threadIdx.x) - 128 * (1 + NQ);
    const int dp = p.d_pad;
    const int cpr = dp >> 3;  // 8-column chunks per f16 row
    // chunk c = row * cpr + ch of a tile, walked as c = tid, tid + 128, ...
    // without a division per chunk: 128 chunks ahead is row_step rows and
    // ch_step chunks further on
    const int row_first = tid / cpr, ch_first = tid - row_first * cpr;
    const int row_step = 128 / cpr, ch_step = 128 - row_step * cpr;
    const int64_t n_bh = p.n_tiles / p.n_qblocks;
    const int64_t n_jobs = n_bh * T;
    const int64_t grid = gridDim.x;
    const int64_t nqb = p.n_qblocks;
    const uint32_t slot = base_s + P::kOffF32 + static_cast<uint32_t>(NQ * P::kF32TileBytes);
    const uint32_t slot_bar = bar(kBarF32Full + NQ);
    if (tid == 0) {
      ptx::prefetch_tensormap(&tm_kl);
      ptx::prefetch_tensormap(&tm_vl);
    }
    // Thread 0 issues each load and waits for it (bounded); the warpgroup
    // learns the outcome through shared memory after a barrier, so that all
    // 128 threads take the same branch and every warpgroup barrier is
    // complete, then each thread acquires the (completed) phase itself.
    volatile uint32_t* conv_ok = reinterpret_cast<volatile uint32_t*>(base + P::kOffBar + kConvOkOff);
    uint32_t loads = 0;  // TMA loads into the slot (thread 0 issues them; phase = loads & 1)
    bool ok = true;
    auto stage = [&](const CUtensorMap* tm, uint16_t* dst, int64_t h, int64_t j, int nr) -> bool {
      const uint32_t phase = loads & 1u;
      ++loads;
      if (tid == 0) {
        ptx::mbar_arrive_expect_tx(slot_bar, P::kF32TileBytes);
        ptx::tma_load_3d_hint(slot, tm, slot_bar, 0, static_cast<int>(j) * kBN,
                              static_cast<int>(h), ptx::policy_evict_first());
        *conv_ok = w.wait(slot_bar, phase, kSiteConvert) ? 1u : 0u;
      }
      ptx::named_barrier_sync(1, 128);
      if (*conv_ok == 0u) return false;
      ptx::mbar_try_wait(slot_bar, phase);  // complete: returns at once, with acquire
      uint16_t* row0 = dst + (h * N + j * kBN) * dp;
      // the f16 rows are read back by every query block of the head: they
      // are the last lines to leave L2 (with the f32 inputs and the output
      // streamed evict-first, the copies are neither re-read from nor, during
      // the call, written back to HBM)
      const uint64_t keep = ptx::policy_evict_last();
      for (int row = row_first, ch = ch_first; row < nr;) {
        const uint32_t a = slot + static_cast<uint32_t>(row * 256 + ch * 32);
        const float4 lo = ptx::ld_shared_v4(a);
        const float4 hi = ptx::ld_shared_v4(a + 16u);
        ptx::st_global_v4_hint(row0 + static_cast<int64_t>(row) * dp + ch * 8,
                               ptx::pack_half2(lo.x, lo.y), ptx::pack_half2(lo.z, lo.w),
                               ptx::pack_half2(hi.x, hi.y), ptx::pack_half2(hi.z, hi.w), keep);
        row += row_step;
        ch += ch_step;
        if (ch >= cpr) {
          ch -= cpr;
          ++row;
        }
      }
      // every thread has read the slot before the next TMA load refills it
      ptx::fence_proxy_async_smem();
      ptx::named_barrier_sync(1, 128);
      return true;
    };
    // The rounds of the job sequence: round r holds the heads [h0, h1) (h0
    // = ceil(r * grid / nqb)), T jobs each, from job base_job on.  A block's
    // jobs increase, so the round is advanced, not searched, per job.
    int64_t r = 0, base_job = 0, h0 = 0;
    int64_t h1 = (grid + nqb - 1) / nqb < n_bh ? (grid + nqb - 1) / nqb : n_bh;
    for (int64_t s = blockIdx.x; ok && s < n_jobs; s += grid) {
      // (bh, j) of job s
      while (s >= base_job + (h1 - h0) * T) {
        base_job += (h1 - h0) * T;
        ++r;
        h0 = h1;
        h1 = ((r + 1) * grid + nqb - 1) / nqb;
        if (h1 > n_bh) h1 = n_bh;
      }
      const int64_t o = s - base_job;
      const int64_t j = o / (h1 - h0);
      const int64_t h = h0 + (o - j * (h1 - h0));
      const int nr = (N - static_cast<int>(j) * kBN) < kBN ? (N - static_cast<int>(j) * kBN) : kBN;
      if (!(ok = stage(&tm_kl, p.k16, h, j, nr))) break;
      if (!(ok = stage(&tm_vl, p.v16, h, j, nr))) break;
      // the copies are read by other blocks through TMA: generic writes,
      // then the proxy fence, the warpgroup barrier and one release
      ptx::fence_proxy_async_global();
      ptx::named_barrier_sync(1, 128);
      if (tid == 0) {
        __threadfence();
        ptx::st_release_gpu(p.kv_ready + h * T + j, 1u);
      }
    }
    // a load still in flight (after an abort) must land before the block exits
    if (tid == 0 && loads > 0) w.drain(slot_bar, (loads - 1) & 1u, kSiteDrainTma);
    (void)ok;
  } else if (convert_wg) {
    if (P::kSplitRegs) ptx::regs_decrease<P::kRegsOther>();
    // ------------------------------------------------ f32 -> f16 converters
    // Ring tile n (slot n % 2) is the n-th of the sequence warp 0 loads; it
    // goes to the K or V stage of its key tile or to a Q tile once the MMAs
    // are done with that buffer.  Warp cw rounds rows [32 cw, 32 cw + 32):
    // per step four rows, 8 lanes per row, eight f32 columns per lane, into
    // one 16-byte unit of the 128-byte-swizzled f16 layout TMA would have
    // written (unit u of row r at u ^ (r & 7)).
    const int cw = warp - (4 + 4 * NQ);
    int64_t n = 0;
    auto convert = [&](uint32_t dst, int full_bar) -> bool {
      const int slot = static_cast<int>(n % kRing);
      if (!w.wait_warp(bar(kBarF32Full + slot), static_cast<uint32_t>((n / kRing) & 1),
                       kSiteConvert))
        return false;
      const uint32_t src = base_s + P::kOffF32 + static_cast<uint32_t>(slot * P::kF32TileBytes);
      const int u = lane & 7;  // f32 columns 8 u .. 8 u + 7 = 16-byte f16 unit u
#pragma unroll 2
      for (int it = 0; it < 8; ++it) {
        const int r = 32 * cw + 4 * it + (lane >> 3);
        const uint32_t a = src + static_cast<uint32_t>(r * 256 + u * 32);
        const float4 x0 = ptx::ld_shared_v4(a);
        const float4 x1 = ptx::ld_shared_v4(a + 16u);
        ptx::st_shared_v4(dst + static_cast<uint32_t>(r * 128 + ((u ^ (r & 7)) << 4)),
                          __uint_as_float(ptx::pack_half2(x0.x, x0.y)),
                          __uint_as_float(ptx::pack_half2(x0.z, x0.w)),
                          __uint_as_float(ptx::pack_half2(x1.x, x1.y)),
                          __uint_as_float(ptx::pack_half2(x1.z, x1.w)));
      }
      ptx::fence_proxy_async_smem();  // the tensor core reads what was written
      __syncwarp();
      if (lane == 0) {
        ptx::mbar_arrive(bar(kBarF32Empty + slot));
        ptx::mbar_arrive(bar(full_bar));
      }
      ++n;
      return true;
    };
    bool ok = true;
    int g = 0;  // key tiles of this block so far
    for (int i = 0; ok && i < n_mine; ++i) {
      const int j0 = sched(i).j0, j1 = sched(i).j1;
      for (int j = j0; ok && j < j1; ++j, ++g) {
        const int st = kv_stage(g);
        const uint32_t free_par = kv_phase(g) ^ 1u;
        if (!(ok = w.wait_warp(bar(kBarKEmpty + st), free_par, kSiteConvert))) break;
        if (!(ok = convert(base_s + P::kOffK + st * P::kStageStride, kBarKFull + st))) break;
        if (!(ok = w.wait_warp(bar(kBarVEmpty + st), free_par, kSiteConvert))) break;
        if (!(ok = convert(base_s + P::kOffV + st * P::kStageStride, kBarVFull + st))) break;
        if (j == j0) {
          // the Q tiles of piece i, once the S products of piece i - 1 are done
          if (i > 0 && !(ok = w.wait_warp(bar(kBarQEmpty), static_cast<uint32_t>(i - 1) & 1u,
                                          kSiteConvert)))
            break;
          for (int t = 0; ok && t < NQ; ++t)
            ok = convert(base_s + P::kOffQ + t * P::kStageStride, kBarQFull);
        }
      }
    }
  } else if (!softmax_wg) {
    if (P::kSplitRegs) ptx::regs_decrease<P::kRegsOther>();
    if (kF32 && warp == 0) {
      // -------------------------------------------------- f32 ring producer
      if (lane == 0) {
        ptx::prefetch_tensormap(&tm_q);
        ptx::prefetch_tensormap(&tm_k);
        ptx::prefetch_tensormap(&tm_v);
        ptx::grid_dep_wait();  // the previous kernel's writes of q, k, v are visible
        int64_t n = 0;
        auto load = [&](const CUtensorMap* tm, int row0, int bh) -> bool {
          const int slot = static_cast<int>(n % kRing);
          if (!w.wait(bar(kBarF32Empty + slot),
                      static_cast<uint32_t>(((n / kRing) & 1) ^ 1), kSiteProducerK))
            return false;
          ptx::mbar_arrive_expect_tx(bar(kBarF32Full + slot), P::kF32TileBytes);
          ptx::tma_load_3d(base_s + P::kOffF32 + static_cast<uint32_t>(slot * P::kF32TileBytes),
                           tm, bar(kBarF32Full + slot), 0, row0, bh);
          ++n;
          return true;
        };
        bool ok = true;
        for (int i = 0; ok && i < n_mine; ++i) {
          const Piece pc = sched(i);
          const int bh = pc.tile / p.n_qblocks;
          const int row0 = (pc.tile % p.n_qblocks) * (kBM * NQ);
          for (int j = pc.j0; ok && j < pc.j1; ++j) {
            ok = load(&tm_k, j * kBN, bh) && load(&tm_v, j * kBN, bh);
            for (int t = 0; ok && j == pc.j0 && t < NQ; ++t)
              ok = load(&tm_q, row0 + t * kBM, bh);
          }
        }
        // every issued copy must have landed before the block exits
        for (int64_t m = (n > kRing ? n - kRing : 0); m < n; ++m)
          w.drain(bar(kBarF32Full + static_cast<int>(m % kRing)),
                  static_cast<uint32_t>((m / kRing) & 1), kSiteDrainTma);
      }
    } else if (warp == 0) {
      // ------------------------------------------------- K/V producer
      // Runs ahead across tile boundaries: the next tile's first K/V tiles
      // are in flight while the current one ends.
      if (lane == 0) {
        ptx::prefetch_tensormap(&tm_k);
        ptx::prefetch_tensormap(&tm_v);
        ptx::grid_dep_wait();  // the previous kernel (the staging pass) has written K and V
        if constexpr (kAcc) {
          ptx::prefetch_tensormap(&tm_kl);
          ptx::prefetch_tensormap(&tm_vl);
        }
        int64_t k_issued = 0, v_issued = 0;
        const uint64_t keep = ptx::policy_evict_last();  // K/V tiles: read by every query block
        bool ok = true;
        int g = 0;  // key tiles of this block so far
        for (int i = 0; ok && i < n_mine; ++i) {
          const Piece pc = sched(i);
          const int bh = pc.tile / p.n_qblocks;
          for (int j = pc.j0; j < pc.j1; ++j, ++g) {
            const int st = kv_stage(g);
            const uint32_t free_par = kv_phase(g) ^ 1u;
            if constexpr (P::kStageKV) {
              // the f16 copies of this key tile are written by a block of
              // this grid: wait for its flag, then read them with TMA
              if (!(ok = w.wait_flag(p.kv_ready + static_cast<int64_t>(bh) * T + j, kSiteKvReady)))
                break;
              ptx::fence_proxy_async_global();
            }
            if (!(ok = w.wait(bar(kBarKEmpty + st), free_par, kSiteProducerK))) break;
            ptx::mbar_arrive_expect_tx(bar(kBarKFull + st), P::kParts * tile_bytes);
            for (int kb = 0; kb < NKB; ++kb) {
              ptx::tma_load_3d_hint(base_s + P::kOffK + st * P::kStageStride + kb * kBoxBytes,
                                    &tm_k, bar(kBarKFull + st), kb * 64, j * kBN, bh, keep);
              if constexpr (kAcc)
                ptx::tma_load_3d(base_s + P::kOffK + st * P::kStageStride + P::kPartBytes +
                                     kb * kBoxBytes,
                                 &tm_kl, bar(kBarKFull + st), kb * 64, j * kBN, bh);
            }
            ++k_issued;
            if (!(ok = w.wait(bar(kBarVEmpty + st), free_par, kSiteProducerV))) break;
            ptx::mbar_arrive_expect_tx(bar(kBarVFull + st), P::kParts * tile_bytes);
            for (int kb = 0; kb < NKB; ++kb) {
              ptx::tma_load_3d_hint(base_s + P::kOffV + st * P::kStageStride + kb * kBoxBytes,
                                    &tm_v, bar(kBarVFull + st), kb * 64, j * kBN, bh, keep);
              if constexpr (kAcc)
                ptx::tma_load_3d(base_s + P::kOffV + st * P::kStageStride + P::kPartBytes +
                                     kb * kBoxBytes,
                                 &tm_vl, bar(kBarVFull + st), kb * 64, j * kBN, bh);
            }
            ++v_issued;
          }
        }
        // every issued copy must have landed before the block exits
        for (int64_t g = (k_issued > S ? k_issued - S : 0); g < k_issued; ++g)
          w.drain(bar(kBarKFull + kv_stage(g)), kv_phase(g), kSiteDrainTma);
        for (int64_t g = (v_issued > S ? v_issued - S : 0); g < v_issued; ++g)
          w.drain(bar(kBarVFull + kv_stage(g)), kv_phase(g), kSiteDrainTma);
      }
    } else if (warp == 3 && P::kF32Q) {
      // ----------------------------------------- Q from f32, rounded here
      // Q_t of tile i comes by TMA into f32 slot t while tile i - 1 runs;
      // once the S products of tile i - 1 are done with the Q tiles, the
      // warp rounds slot t into Q tile t (four rows per step, 8 lanes per
      // row, eight f32 columns per lane, one 16-byte unit of the
      // 128-byte-swizzled f16 layout each), tells the S issuer that tile t
      // is ready and reloads slot t with the next tile's Q_t.
      auto load_q = [&](int i, int t) {
        ptx::mbar_arrive_expect_tx(bar(kBarF32Full + t), P::kF32TileBytes);
        ptx::tma_load_3d_hint(base_s + P::kOffF32 + static_cast<uint32_t>(t * P::kF32TileBytes),
                              &tm_q, bar(kBarF32Full + t), 0, tile_row0(i) + t * kBM, tile_bh(i),
                              ptx::policy_evict_first());  // each q row is read once
      };
      if (lane == 0) {
        ptx::prefetch_tensormap(&tm_q);
        ptx::grid_dep_wait();
        for (int t = 0; t < NQ; ++t) load_q(0, t);
      }
      int q_loaded[NQ];  // per slot: tiles whose Q load was issued (lane 0)
      for (int t = 0; t < NQ; ++t) q_loaded[t] = 1;
      bool ok = true;
      const int u = lane & 7;  // f32 columns 8 u .. 8 u + 7 = 16-byte f16 unit u
      for (int i = 0; ok && i < n_mine; ++i) {
        if (i > 0 && !(ok = w.wait_warp(bar(kBarQEmpty), static_cast<uint32_t>(i - 1) & 1u,
                                        kSiteProducerQ)))
          break;
        for (int t = 0; ok && t < NQ; ++t) {
          if (!(ok = w.wait_warp(bar(kBarF32Full + t), static_cast<uint32_t>(i) & 1u, kSiteConvert)))
            break;
          const uint32_t src = base_s + P::kOffF32 + static_cast<uint32_t>(t * P::kF32TileBytes);
          const uint32_t dst = base_s + P::kOffQ + static_cast<uint32_t>(t * P::kStageStride);
#pragma unroll 4
          for (int it = 0; it < kBM / 4; ++it) {
            const int r = 4 * it + (lane >> 3);
            const uint32_t a = src + static_cast<uint32_t>(r * 256 + u * 32);
            const float4 x0 = ptx::ld_shared_v4(a);
            const float4 x1 = ptx::ld_shared_v4(a + 16u);
            ptx::st_shared_v4(dst + static_cast<uint32_t>(r * 128 + ((u ^ (r & 7)) << 4)),
                              __uint_as_float(ptx::pack_half2(x0.x, x0.y)),
                              __uint_as_float(ptx::pack_half2(x0.z, x0.w)),
                              __uint_as_float(ptx::pack_half2(x1.x, x1.y)),
                              __uint_as_float(ptx::pack_half2(x1.z, x1.w)));
          }
          // the tensor core reads Q tile t, and the next TMA writes slot t,
          // after this warp's shared-memory accesses
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            ptx::mbar_arrive(bar(t == 0 ? kBarQFull : kBarQFull1));
            if (i + 1 < n_mine) {
              load_q(i + 1, t);
              ++q_loaded[t];
            }
          }
        }
      }
      // every issued copy must have landed before the block exits
      if (lane == 0)
        for (int t = 0; t < NQ; ++t)
          w.drain(bar(kBarF32Full + t), static_cast<uint32_t>(q_loaded[t] - 1) & 1u, kSiteDrainTma);
    } else if (warp == 3 && !kF32) {
      // --------------------------------------------------- Q producer
      // The Q tiles of tile i go in as soon as the S products of tile i-1
      // have read the previous ones.
      if (lane == 0) {
        ptx::prefetch_tensormap(&tm_q);
        if constexpr (kAcc) ptx::prefetch_tensormap(&tm_ql);
        ptx::grid_dep_wait();  // ... and Q
        int q_issued = 0;
        for (int i = 0; i < n_mine; ++i) {
          if (i > 0 && !w.wait(bar(kBarQEmpty), static_cast<uint32_t>(i - 1) & 1u, kSiteProducerQ))
            break;
          ptx::mbar_arrive_expect_tx(bar(kBarQFull), NQ * P::kParts * tile_bytes);
          for (int t = 0; t < NQ; ++t)
            for (int kb = 0; kb < NKB; ++kb) {
              ptx::tma_load_3d(base_s + P::kOffQ + t * P::kStageStride + kb * kBoxBytes, &tm_q,
                               bar(kBarQFull), kb * 64, tile_row0(i) + t * kBM, tile_bh(i));
              if constexpr (kAcc)
                ptx::tma_load_3d(base_s + P::kOffQ + t * P::kStageStride + P::kPartBytes +
                                     kb * kBoxBytes,
                                 &tm_ql, bar(kBarQFull), kb * 64, tile_row0(i) + t * kBM,
                                 tile_bh(i));
            }
          ++q_issued;
        }
        if (q_issued > 0)
          w.drain(bar(kBarQFull), static_cast<uint32_t>(q_issued - 1) & 1u, kSiteDrainTma);
      }
    } else if (warp == 1 || warp == 2) {
      // ---------------------------------------------------------- MMA issuers
      // Two threads issue tcgen05.mma: the S products depend on the softmax
      // having copied S out, the P V products on P being written, and on
      // nothing else of each other, so each issuer waits once per key tile.
      if (lane == 0 && warp == 1) {
        // S(t, g) = Q_t K_g^T into S buffer sbuf(t, g)
        const uint32_t idesc_s = ptx::idesc_f16_f32(kBM, kBN, false);
        const int ksteps = p.d_pad >> 4;
        auto issue_s = [&](int t, int64_t g) {
          const uint32_t qa = base_s + P::kOffQ + t * P::kStageStride;
          const uint32_t kb = base_s + P::kOffK + kv_stage(g) * P::kStageStride;
          const uint32_t d = tmem + static_cast<uint32_t>(sbuf(t, g)) * 128u;
          if constexpr (!kAcc && NKB == 1) {
            if (ksteps == 4) {
              // head_dim 49..64: the descriptors as 32-bit halves, one add per
              // product (fewer instructions between the blocking issues)
              constexpr uint32_t hi = ptx::smem_desc_hi(1024, ptx::kSwizzle128B);
              const uint32_t qlo = ptx::smem_desc_lo(qa, 16), klo = ptx::smem_desc_lo(kb, 16);
#pragma unroll
              for (int ks = 0; ks < 4; ++ks)
                ptx::mma_ss(d, ptx::smem_desc_join(qlo + 2u * ks, hi),
                            ptx::smem_desc_join(klo + 2u * ks, hi), idesc_s, ks > 0 ? 1u : 0u);
              ptx::mma_commit(bar(kBarSFull + sbuf(t, g)));
              return;
            }
          }
          for (int ks = 0; ks < ksteps; ++ks) {
            const uint32_t off = static_cast<uint32_t>((ks >> 2) * kBoxBytes + (ks & 3) * 32);
            ptx::mma_ss(d, ptx::smem_desc(qa + off, 16, 1024, ptx::kSwizzle128B),
                        ptx::smem_desc(kb + off, 16, 1024, ptx::kSwizzle128B), idesc_s,
                        ks > 0 ? 1u : 0u);
            if constexpr (kAcc) {  // + Qh Kl^T + Ql Kh^T
              ptx::mma_ss(d, ptx::smem_desc(qa + off, 16, 1024, ptx::kSwizzle128B),
                          ptx::smem_desc(kb + P::kPartBytes + off, 16, 1024, ptx::kSwizzle128B),
                          idesc_s, 1u);
              ptx::mma_ss(d, ptx::smem_desc(qa + P::kPartBytes + off, 16, 1024, ptx::kSwizzle128B),
                          ptx::smem_desc(kb + off, 16, 1024, ptx::kSwizzle128B), idesc_s, 1u);
            }
          }
          ptx::mma_commit(bar(kBarSFull + sbuf(t, g)));
        };
        bool ok = true;
        int g = 0;  // key tiles of this block so far
        for (int i = 0; ok && i < n_mine; ++i) {
          if (!(ok = w.wait(bar(kBarQFull), static_cast<uint32_t>(i) & 1u, kSiteMmaQ))) break;
          const Piece pc = sched(i);
          for (int j = pc.j0; j < pc.j1; ++j, ++g) {
            // S of key tile g needs K_g and the softmax to have copied the
            // previous contents of its buffer(s) to registers
            if (!(ok = w.wait(bar(kBarKFull + kv_stage(g)), kv_phase(g), kSiteMmaK))) break;
            const int prev = NQ == 2 ? g - 1 : g - 2;  // last key tile that used the buffer(s)
            if (prev >= 0 &&
                !(ok = w.wait(bar(kBarSFree + sfree_bar(prev)), sphase(prev), kSiteMmaSFree)))
              break;
            ptx::tc_fence_after();
            for (int t = 0; t < NQ; ++t) {
              if (P::kF32Q && j == pc.j0 && t == 1) {  // Q tile 1 is rounded after tile 0
                if (!(ok = w.wait(bar(kBarQFull1), static_cast<uint32_t>(i) & 1u, kSiteMmaQ))) break;
                ptx::tc_fence_after();
              }
              issue_s(t, g);
            }
            if (!ok) break;
            ptx::mma_commit(bar(kBarKEmpty + kv_stage(g)));
          }
          // the Q tiles are free once these S products have run
          if (ok) ptx::mma_commit(bar(kBarQEmpty));
        }
        ptx::mma_commit(bar(kBarMmaDone));
      } else if (lane == 0 && warp == 2) {
        // O_t += P_t V_g
        const uint32_t idesc_pv = ptx::idesc_f16_f32(kBM, static_cast<uint32_t>(p.d_pad), true);
        // k-steps [ks0, ks1) of O_t += P_t V_g, then a commit on `done`
        auto issue_pv = [&](int t, int64_t g, bool first, int ks0, int ks1, int done) {
          const uint32_t vb = base_s + P::kOffV + kv_stage(g) * P::kStageStride;
          const uint32_t d = tmem + P::kColO + static_cast<uint32_t>(t) * P::kColOStride;
          const uint32_t a = tmem + P::kColP + static_cast<uint32_t>(t) * P::kColPStride;
          if constexpr (!kAcc) {
            // the V descriptor as 32-bit halves, one add per product (fewer
            // instructions between the blocking issues); k-step ks starts
            // 16 rows (2048 bytes) further on
            constexpr uint32_t hi = ptx::smem_desc_hi(1024, ptx::kSwizzle128B);
            const uint32_t vlo = ptx::smem_desc_lo(vb, kBoxBytes);
            for (int ks = ks0; ks < ks1; ++ks)
              ptx::mma_ts(d, a + static_cast<uint32_t>(ks) * 8u,
                          ptx::smem_desc_join(vlo + static_cast<uint32_t>(ks) * (2048u >> 4), hi),
                          idesc_pv, (!first || ks > 0) ? 1u : 0u);
          } else {
            for (int ks = ks0; ks < ks1; ++ks) {  // Ph Vh + Ph Vl + Pl Vh
              ptx::mma_ts(d, a + static_cast<uint32_t>(ks) * 8u,
                          ptx::smem_desc(vb + ks * 2048, kBoxBytes, 1024, ptx::kSwizzle128B),
                          idesc_pv, (!first || ks > 0) ? 1u : 0u);
              ptx::mma_ts(d, a + static_cast<uint32_t>(ks) * 8u,
                          ptx::smem_desc(vb + P::kPartBytes + ks * 2048, kBoxBytes, 1024,
                                         ptx::kSwizzle128B),
                          idesc_pv, 1u);
              ptx::mma_ts(d, tmem + P::kColPlo + static_cast<uint32_t>(ks) * 8u,
                          ptx::smem_desc(vb + ks * 2048, kBoxBytes, 1024, ptx::kSwizzle128B),
                          idesc_pv, 1u);
            }
          }
          ptx::mma_commit(bar(done));
        };
        bool ok = true;
        int g = 0;  // key tiles of this block so far
        for (int i = 0; ok && i < n_mine; ++i) {
          const Piece pc = sched(i);
          for (int j = pc.j0; j < pc.j1; ++j, ++g) {
            if (!(ok = w.wait(bar(kBarVFull + kv_stage(g)), kv_phase(g), kSiteMmaV))) break;
            // P of key tile g written (for the first key tile of a tile this
            // also tells that the softmax has read the previous tile's O)
            if constexpr (P::kSharedP) {
              // the two query tiles take turns with the P buffer, half by
              // half: tile t's first half (keys 0..63) goes to the tensor
              // core as soon as it is written, while the softmax writes the
              // second half once the other tile's P V has read it
              for (int t = 0; ok && t < NQ; ++t) {
                if (!(ok = w.wait(bar(kBarPHalf + t), static_cast<uint32_t>(g & 1), kSiteMmaP))) break;
                ptx::tc_fence_after();
                issue_pv(t, g, j == pc.j0, 0, kBN / 32, kBarOHalf + t);
                if (!(ok = w.wait(bar(kBarPFull + t), static_cast<uint32_t>(g & 1), kSiteMmaP))) break;
                ptx::tc_fence_after();
                issue_pv(t, g, j == pc.j0, kBN / 32, kBN / 16, kBarODone + t);
              }
              if (!ok) break;
            } else {
              if (!(ok = w.wait(bar(kBarPFull), static_cast<uint32_t>(g & 1), kSiteMmaP))) break;
              ptx::tc_fence_after();
              for (int t = 0; t < NQ; ++t) issue_pv(t, g, j == pc.j0, 0, kBN / 16, kBarODone + t);
            }
            ptx::mma_commit(bar(kBarVEmpty + kv_stage(g)));
          }
        }
        ptx::mma_commit(bar(kBarMmaDone));
      }
    }
  } else {
    if (P::kSplitRegs) ptx::regs_increase<P::kRegsSoftmax>();
    // ------------------------------------------------------------ softmax
    const int t = (warp - 4) >> 2;
    const int quarter = warp & 3;
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t p_addr = tmem + lane_addr + P::kColP + static_cast<uint32_t>(t) * P::kColPStride;
    const uint32_t o_addr = tmem + lane_addr + P::kColO + static_cast<uint32_t>(t) * P::kColOStride;
    bool ok = true;
    int g = 0;  // key tiles of this block so far
    for (int i = 0; ok && i < n_mine; ++i) {
      const int j0 = sched(i).j0, j1 = sched(i).j1;
      float m_ref = -INFINITY;  // running max in log2 units (may lag the true max by < 8)
      float l = 0.0f;           // running sum of exp2(s*log2e - m_ref)
      for (int j = j0; j < j1; ++j, ++g) {
        const int buf = sbuf(t, g);
        if (!(ok = w.wait_warp(bar(kBarSFull + buf), sphase(g), kSiteSoftS))) break;
        ptx::tc_fence_after();
        const uint32_t s_addr = tmem + lane_addr + static_cast<uint32_t>(buf) * 128u;
        const int valid = N - j * kBN;

        // the whole S row (128 columns) into registers, one wait; then the
        // buffer is released for the next S = Q K^T
        uint32_t r[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) ptx::tmem_ld_32x32b_x32(s_addr + c * 32, r[c]);
#pragma unroll
        for (int c = 0; c < 4; ++c) ptx::tmem_wait_ld_dep(r[c]);
        ptx::tc_fence_before();
        warp_arrive(bar(kBarSFree + sfree_bar(g)));

        if (valid < kBN) {  // ragged last key tile only: keys >= n_patches score -inf
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (c * 32 + e >= valid) r[c][e] = 0xff800000u;
        }
        float mc[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float a = -INFINITY;
#pragma unroll
          for (int e = 0; e < 32; e += 2)
            a = ptx::max3(a, __uint_as_float(r[c][e]), __uint_as_float(r[c][e + 1]));
          mc[c] = a;
        }
        const float mt = ptx::max3(mc[0], mc[1], fmaxf(mc[2], mc[3])) * kLog2e;
        const bool need = mt > m_ref + kRescaleLog2;
        const float m_new = need ? mt : m_ref;
        const float alpha = ptx::ex2_approx(m_ref - m_new);  // 0 on the first key tile, 1 if kept
        m_ref = m_new;

        // p = 2^(s*log2e - m_ref) as f16 pairs, kept in registers: the P
        // buffer may still be read by the previous key tile's P V, which
        // runs on the tensor core meanwhile
        const float2 scale = make_float2(kLog2e, kLog2e);
        const float2 shift = make_float2(-m_ref, -m_ref);
        float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                         make_float2(0.f, 0.f)};
        uint32_t pk[4][16];
        uint32_t pkl[kAcc ? 4 : 1][16];  // accurate mode: P lo = f16(p - f32(P hi))
#pragma unroll
        for (int c = 0; c < 4; ++c) {
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float2 x = __ffma2_rn(
                make_float2(__uint_as_float(r[c][2 * e]), __uint_as_float(r[c][2 * e + 1])), scale,
                shift);
            const float2 pp = make_float2(ptx::ex2_approx(x.x), ptx::ex2_approx(x.y));
            acc[e & 3] = __fadd2_rn(acc[e & 3], pp);
            pk[c][e] = ptx::pack_half2(pp.x, pp.y);
            if constexpr (kAcc) {
              const float2 back = __half22float2(*reinterpret_cast<const __half2*>(&pk[c][e]));
              pkl[c][e] = ptx::pack_half2(pp.x - back.x, pp.y - back.y);
            }
          }
        }
        const float2 s01 = __fadd2_rn(acc[0], acc[1]);
        const float2 s23 = __fadd2_rn(acc[2], acc[3]);
        l = fmaf(l, alpha, (s01.x + s01.y) + (s23.x + s23.y));
        const int64_t gw = t == 0 ? g - 1 : g;  // shared P: the other tile's P V before ours
        if (P::kSharedP) {
          // one P buffer, used by (tile 0, g), (tile 1, g), (tile 0, g + 1), ...,
          // half by half: tile 0 writes its first half once the P V of (1,
          // g - 1) has read that half, tile 1 once that of (0, g) has.  One
          // thread issues the products in that order and a commit tracks all
          // earlier ones, so this also means the tile's own previous P V has
          // finished (O final for a rescale).
          if (gw >= 0) {
            if (!(ok = w.wait_warp(bar(kBarOHalf + (1 - t)), static_cast<uint32_t>(gw & 1),
                                   kSiteSoftO)))
              break;
            ptx::tc_fence_after();
          }
        } else if (j > j0) {
          // P V of the previous key tile has finished: P buffer free, O final.
          // (For a piece's first key tile the previous epilogue waited for it.)
          if (!(ok = w.wait_warp(bar(kBarODone + t), static_cast<uint32_t>((g - 1) & 1),
                                 kSiteSoftO)))
            break;
          ptx::tc_fence_after();
        }
        if (j > j0) {
          if (__any_sync(0xffffffffu, need)) {
            for (int c = 0; c < (p.d_pad >> 4); ++c) {
              uint32_t y[16];
              ptx::tmem_ld_32x32b_x16(o_addr + c * 16, y);
              ptx::tmem_wait_ld_dep16(y);
#pragma unroll
              for (int e = 0; e < 16; ++e) y[e] = __float_as_uint(__uint_as_float(y[e]) * alpha);
              ptx::tmem_st_32x32b_x16(o_addr + c * 16, y);
            }
          }
        }
        if constexpr (P::kSharedP) {
          // first half, then (once the other tile's P V has read the whole
          // buffer) the second half
#pragma unroll
          for (int c = 0; c < 2; ++c) ptx::tmem_st_32x32b_x16(p_addr + c * 16, pk[c]);
          ptx::tmem_wait_st();
          ptx::tc_fence_before();
          warp_arrive(bar(kBarPHalf + t));
          if (gw >= 0) {
            if (!(ok = w.wait_warp(bar(kBarODone + (1 - t)), static_cast<uint32_t>(gw & 1),
                                   kSiteSoftO)))
              break;
            ptx::tc_fence_after();
          }
#pragma unroll
          for (int c = 2; c < 4; ++c) ptx::tmem_st_32x32b_x16(p_addr + c * 16, pk[c]);
          ptx::tmem_wait_st();
          ptx::tc_fence_before();
          warp_arrive(bar(kBarPFull + t));
        } else {
#pragma unroll
          for (int c = 0; c < 4; ++c) ptx::tmem_st_32x32b_x16(p_addr + c * 16, pk[c]);
          if constexpr (kAcc) {
#pragma unroll
            for (int c = 0; c < 4; ++c)
              ptx::tmem_st_32x32b_x16(tmem + lane_addr + P::kColPlo + c * 16, pkl[c]);
          }
          ptx::tmem_wait_st();
          ptx::tc_fence_before();
          warp_arrive(bar(kBarPFull));
        }
      }
      if (!ok) break;
      // ---- epilogue of the tile: out = O / l for the rows < n_patches.  The
      // next tile's first P V overwrites O only after this warp's next P
      // arrival, which follows these reads.
      if (!(ok = w.wait_warp(bar(kBarODone + t), static_cast<uint32_t>((g - 1) & 1),
                             kSiteEpilogue)))
        break;
      ptx::tc_fence_after();
      const Piece pc = sched(i);
      if (pc.slot >= 0) {
        // A tile cut between two neighbouring blocks (keys [0, c) in one,
        // [c, T) in the other).  The part that ends first leaves its O
        // (unnormalised), m and l in the slot and raises the slot's flag; the
        // part that ends second waits for the flag (the other part is then
        // already writing it), adds the partial into its own O by the
        // log-sum-exp rule -- the shader's rescale of (m, l, o) by the
        // larger of the two maxima -- and stores the tile as usual.
        // Each warp (its 32 rows) meets its counterpart on its own: arrival
        // count and flag per (slot, query tile, warp), no block-wide barrier.
        const size_t slot_floats = static_cast<size_t>(kBM) * static_cast<size_t>(p.d_pad + 2);
        float* part = p.part + (static_cast<size_t>(pc.slot) * NQ + t) * slot_floats;
        float4* part4 = reinterpret_cast<float4*>(part);  // column group c4 of row r at c4 * 128 + r
        uint32_t* sync = p.part_sync + ((static_cast<size_t>(pc.slot) * NQ + t) * 4 + quarter) * 2;
        uint32_t order = 0;
        if (lane == 0) order = atomicAdd(sync, 1u);
        const bool second = __shfl_sync(0xffffffffu, order, 0) != 0u;
        const int r = quarter * 32 + lane;
        if (!second) {
          for (int c = 0; c < (p.d_pad >> 4); ++c) {
            uint32_t y[16];
            ptx::tmem_ld_32x32b_x16(o_addr + c * 16, y);
            ptx::tmem_wait_ld_dep16(y);
#pragma unroll
            for (int k = 0; k < 4; ++k)
              part4[(c * 4 + k) * kBM + r] =
                  make_float4(__uint_as_float(y[4 * k]), __uint_as_float(y[4 * k + 1]),
                              __uint_as_float(y[4 * k + 2]), __uint_as_float(y[4 * k + 3]));
          }
          part[kBM * p.d_pad + r] = m_ref;
          part[kBM * (p.d_pad + 1) + r] = l;
          __threadfence();
          __syncwarp();
          if (lane == 0) ptx::st_release_gpu(sync + 1, 1u);
          ptx::tc_fence_before();
          continue;
        }
        if (!(ok = __all_sync(0xffffffffu, w.wait_flag(sync + 1, kSitePartial)))) break;
        const float mp = part[kBM * p.d_pad + r];
        const float lp = part[kBM * (p.d_pad + 1) + r];
        const float mx = fmaxf(m_ref, mp);
        const float ca = ptx::ex2_approx(m_ref - mx);
        const float cb = ptx::ex2_approx(mp - mx);
        l = ca * l + cb * lp;
        for (int c = 0; c < (p.d_pad >> 4); ++c) {
          uint32_t y[16];
          ptx::tmem_ld_32x32b_x16(o_addr + c * 16, y);
          ptx::tmem_wait_ld_dep16(y);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float4 z = part4[(c * 4 + k) * kBM + r];
            y[4 * k + 0] = __float_as_uint(fmaf(__uint_as_float(y[4 * k + 0]), ca, z.x * cb));
            y[4 * k + 1] = __float_as_uint(fmaf(__uint_as_float(y[4 * k + 1]), ca, z.y * cb));
            y[4 * k + 2] = __float_as_uint(fmaf(__uint_as_float(y[4 * k + 2]), ca, z.z * cb));
            y[4 * k + 3] = __float_as_uint(fmaf(__uint_as_float(y[4 * k + 3]), ca, z.w * cb));
          }
          ptx::tmem_st_32x32b_x16(o_addr + c * 16, y);
        }
        ptx::tmem_wait_st();
      }
      const float inv_l = 1.0f / l;
      if (P::kEpiBytes > 0 && p.tma_out) {
        // 16 columns at a time: TMEM -> registers -> swizzled shared buffer
        // -> one TMA store of the warp's 32 rows (rows past n_patches and
        // columns past head_dim are not written); the stores complete in
        // the background while the warp moves on to the next tile
        const uint32_t epi =
            base_s + P::kOffEpi + static_cast<uint32_t>(warp - 4) * 4096u;
        const int pc_bh = pc.tile / p.n_qblocks;
        const int row_base = (pc.tile % p.n_qblocks) * (kBM * NQ) + t * kBM + quarter * 32;
        for (int c = 0; c < (p.d_pad >> 4); ++c) {
          uint32_t y[16];
          ptx::tmem_ld_32x32b_x16(o_addr + c * 16, y);
          // buffer c & 1 is free once the store issued two chunks earlier
          // (of this tile or the previous one) has read it
          if (lane == 0) ptx::bulk_wait_group_read<1>();
          __syncwarp();
          ptx::tmem_wait_ld_dep16(y);
          const uint32_t buf = epi + static_cast<uint32_t>(c & 1) * 2048u;
          if constexpr (kOut16) {
            // 32 bytes per row, 32-byte swizzle (16-byte unit k at k ^ ((row >> 2) & 1))
            const uint32_t row_addr = buf + static_cast<uint32_t>(lane) * 32u;
#pragma unroll
            for (int k = 0; k < 2; ++k) {
              uint32_t h[4];
#pragma unroll
              for (int e = 0; e < 4; ++e)
                h[e] = ptx::pack_half2(__uint_as_float(y[8 * k + 2 * e]) * inv_l,
                                       __uint_as_float(y[8 * k + 2 * e + 1]) * inv_l);
              ptx::st_shared_v4(row_addr + ((static_cast<uint32_t>(k) ^ ((lane >> 2) & 1u)) << 4),
                                __uint_as_float(h[0]), __uint_as_float(h[1]),
                                __uint_as_float(h[2]), __uint_as_float(h[3]));
            }
          } else {
            const uint32_t row_addr = buf + static_cast<uint32_t>(lane) * 64u;
#pragma unroll
            for (int k = 0; k < 4; ++k)
              ptx::st_shared_v4(row_addr + ((static_cast<uint32_t>(k) ^ ((lane >> 1) & 3u)) << 4),
                                __uint_as_float(y[4 * k + 0]) * inv_l,
                                __uint_as_float(y[4 * k + 1]) * inv_l,
                                __uint_as_float(y[4 * k + 2]) * inv_l,
                                __uint_as_float(y[4 * k + 3]) * inv_l);
          }
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            ptx::tma_store_3d_hint(&tm_o, buf, c * 16, row_base, pc_bh,
                                   ptx::policy_evict_first());  // written once, not read here
            ptx::bulk_commit_group();
          }
        }
        ptx::tc_fence_before();
        continue;
      }
      const int row = (pc.tile % p.n_qblocks) * (kBM * NQ) + t * kBM + quarter * 32 + lane;
      const int pc_bh = pc.tile / p.n_qblocks;
      const int D = p.head_dim;
      if constexpr (kOut16) {
        uint16_t* orow16 = p.out16 + (static_cast<size_t>(pc_bh) * N + row) * D;
        for (int c = 0; c < (p.d_pad >> 4); ++c) {
          uint32_t y[16];
          ptx::tmem_ld_32x32b_x16(o_addr + c * 16, y);
          ptx::tmem_wait_ld_dep16(y);
          if (row < N) {
#pragma unroll
            for (int e = 0; e < 16; e += 2) {
              const int d = c * 16 + e;
              const uint32_t h = ptx::pack_half2(__uint_as_float(y[e]) * inv_l,
                                                 __uint_as_float(y[e + 1]) * inv_l);
              if (d < D) orow16[d] = static_cast<uint16_t>(h & 0xFFFFu);
              if (d + 1 < D) orow16[d + 1] = static_cast<uint16_t>(h >> 16);
            }
          }
        }
        ptx::tc_fence_before();
        continue;
      }
      float* orow = p.out + (static_cast<size_t>(pc_bh) * N + row) * D;
      for (int c = 0; c < (p.d_pad >> 4); ++c) {
        uint32_t y[16];
        ptx::tmem_ld_32x32b_x16(o_addr + c * 16, y);
        ptx::tmem_wait_ld_dep16(y);
        if (row < N) {
          if (p.vec_out) {
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4) {
              const int d = c * 16 + v4 * 4;
              if (d < D) {
                float4 o;
                o.x = __uint_as_float(y[4 * v4 + 0]) * inv_l;
                o.y = __uint_as_float(y[4 * v4 + 1]) * inv_l;
                o.z = __uint_as_float(y[4 * v4 + 2]) * inv_l;
                o.w = __uint_as_float(y[4 * v4 + 3]) * inv_l;
                *reinterpret_cast<float4*>(orow + d) = o;
              }
            }
          } else {
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const int d = c * 16 + e;
              if (d < D) orow[d] = __uint_as_float(y[e]) * inv_l;
            }
          }
        }
      }
      ptx::tc_fence_before();
    }
    // the output stores must have completed before the block exits
    if (P::kEpiBytes > 0 && p.tma_out && lane == 0) ptx::bulk_wait_group_all();
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    if (lane == 0) w.drain(bar(kBarMmaDone), 0, kSiteDrainMma);
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace vattn
