// Small-M (decode) indexed W4A16 MoE GEMM: weight streaming with register MMA.
//
// [Humming] "워크로드별 튜닝 및 JIT 컴파일": at small batch a multistage
// async-copy + MMA pipeline beats TMA + UMMA; [Chord] "인덱스 커널 기법":
// decode is a weight-streaming problem.  Design on sm_103a:
//   * persistent CTAs (as many as fit: 4 per SM for 8 rows per pass) take
//     work items from a global counter: item = (64-row weight tile, BLOCK_M
//     block of the aligned rows), block index fastest, read through the
//     align buffers (expert_ids, num_tokens_post_padded); the blocks of a
//     heavy expert become separate items that stream the same tile together
//     (L2 hits), and the tail is one small item; the last CTA to run dry
//     zeroes the counter;
//   * one producer warp issues 1-D bulk async copies (TMA engine) of the
//     contiguous packed units and of the block's activation rows into a
//     2-stage shared-memory ring of 512 of K per stage, completing on
//     mbarriers (two large stages beat four small ones: each stage hand-off
//     costs several hundred cycles, so fewer hand-offs per byte win: 2 x 8
//     units measured 8 % faster than 4 x 4 and 6 x 2 40 % slower, in the
//     same shared memory); items flow to the consumers through a small
//     mbarrier-guarded ring;
//   * four consumer warps, one 16-row slab each, decode INT4 nibbles straight
//     into m16n8k16 A fragments (the packed order is the fragment order),
//     take B fragments with ldmatrix, and run mma.sync with weights as the M
//     side and tokens as N ("swap AB");
//   * decoding is one shift and one LOP3 per register, giving q + 136 as a
//     BF16 pair (exact), then one packed BF16 add of -136 giving q exactly
//     (the result is a small integer, so the add does not round); the MMA
//     chain of a 32-wide scale group therefore yields sum(q * x) from exact
//     products, and the group's scale is applied in FP32 (no rounding of
//     q * s).  The packed add runs on the FMA pipe, which is lightly used
//     here; an earlier form kept q + 136 and seeded each chain with
//     -136 * sum(x) by two extra MMAs on the busier tensor pipe, and was
//     5-12 % slower;
//   * epilogue: SiLU(gate) * up (a gate/up slab holds gate rows g and up rows
//     g + 8 of the same intermediate index, so both land in one thread), a
//     plain store, BF16, rows in sorted order, or the weighted add (FP32
//     atomic adds of topk_weights[f] * acc into the token's row);
//   * split-K, gated on grid saturation ([Chord] "인덱스 커널 기법": stream-K
//     only where the grid is not already full): when a launch has at most
//     half as many items as resident CTAs (a few decode tokens touching one
//     or two experts), every item is split into S <= 8 ranges of K stages so
//     that all CTAs stream weights.  Otherwise, when the last, partial wave
//     (n mod CTAs of n items, handed out last) fills more than half of the
//     CTAs, its items are split, into as many ranges as make that wave
//     shortest, so the launch does not end on a whole item's time with its
//     CTAs sharing the SMs.  Each split writes its FP32 partial
//     accumulators to the workspace; the last split of an item to arrive
//     (per-item counters, reset by that last arrival) adds the S partials in
//     split order, so the result does not depend on which CTA finishes last,
//     and runs the epilogue.  The decision is taken on the device from the
//     block count, so it needs no host synchronisation.
#include "common.cuh"
#include "kernels.h"

namespace chord {
namespace {

constexpr int kConsumerWarps = kSlabs;                     // one slab per warp
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kUnitsPerStage = 8;                          // 512 of K per stage
constexpr int kXRowBytes = kUnitsPerStage * kUnitK * 2;    // 512
constexpr int kXPitch = kXRowBytes + 16;                   // conflict-free ldmatrix rows

template <int NT>
struct SmallCfg {
  static constexpr int kRowsPerPass = NT * 8;
  static constexpr int kWBytes = kUnitsPerStage * kUnitBytes;
  static constexpr int kXBytes = kRowsPerPass * kXPitch;
  static constexpr int kStageBytes = kWBytes + kXBytes;
  // FP32 partial accumulators of one split of one item (every consumer lane's)
  static constexpr int kSlotFloats = kConsumerWarps * 32 * 4 * NT;
  static constexpr long long kSlots = static_cast<long long>(kSplitPartialBytes / sizeof(float) / kSlotFloats);
};

constexpr int kItemSlots = 4;
constexpr int kMaxSplit = 8;

// A work item as the producer hands it to the consumers.  rows = -1: end.
struct SItem {
  int tile, e, row0, rows;   // first 64-row weight tile, local expert, first sorted row, rows of the block
  int ntl;                   // consecutive weight tiles in the item (several only when K fits one stage)
  int ks0, ks1;              // K stages [ks0, ks1) of this split
  int slot;                  // split items: partials at slots [slot * S, slot * S + S), counters of slot
  int split;                 // split index | (number of splits S << 16)
};

// How a launch's items split along K: every item into `all` ranges, or the
// items from `head` on into `tail` ranges each (1: no split).
struct SplitPlan {
  int all, tail;
  long long head;
};

struct SmallArgs {
  const uint16_t* A;
  const uint8_t* packed;
  const int32_t* sorted;
  const int32_t* expert_ids;
  const int32_t* ntpp;
  const int32_t* counts;
  const int32_t* offsets;
  int* work;        // [0] next item, [1] CTAs done; zero before the launch, zero after it
  int block_m;
  uint16_t* C;
  float* Cf;             // weighted add: FP32 [M, N] accumulator
  const float* topk_w;   // weighted add: routing weights [M, topk]
  int* status;
  int N, K, M, topk, ldc, n_tiles, E_local;
  int pdl, max_blocks;   // programmatic-launch mode (GemmLaunch::pdl); capacity / block_m
  uint32_t wait_polls;   // probes per main-loop barrier wait (drains always use kWaitPolls)
  int test_timeout;      // test hook: hand out no item, so the consumers' waits run out
  float* partial;        // split-K partial accumulators (kSplitSlots slots); NULL: no split-K
  int* split_cnt;        // per (item, consumer warp) arrival counters, zero between launches
  int64_t tile_bytes;
  uint32_t need_flags;
  // decode constants, passed at run time so they stay in registers
  uint32_t nib_mask, nib_magic, neg136;
};

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

__device__ __forceinline__ float silu_f32(float z) { return z / (1.0f + __expf(-z)); }

__device__ bool header_ok(const SmallArgs& a) {
  const PackHeader* h = reinterpret_cast<const PackHeader*>(a.packed);
  return h->magic == kPackMagic && h->version == kPackVersion && h->N == a.N && h->K == a.K &&
         h->group == kGroup && h->E >= a.E_local && h->tile_bytes == a.tile_bytes &&
         (h->flags & a.need_flags) == a.need_flags;
}

// One 64-wide K unit for one warp's slab and NT token tiles.  Per 32-wide
// group: the MMA chain starts from zero and adds q*x over the group's two
// k16 steps, giving sum(q*x) from exact products; then acc += scale * chain
// in FP32.  Every token tile is computed (columns of
// unused tokens are discarded by the epilogue), so no MMA is predicated.
template <int NT>
__device__ __forceinline__ void unit_mma(uint32_t ub, uint32_t xu, uint32_t q_off, uint32_t s_off,
                                         const SmallArgs& a, float (&acc)[NT][4]) {
  const uint4 q = lds128(ub + q_off);
  const uint2 sc = lds64(ub + s_off);
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    uint32_t bf[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n) ldmatrix_x4(bf[n], xu + n * 8 * kXPitch + half * 64);
    uint32_t a0[4], a1[4];
    decode_word_offset136(half ? q.z : q.x, a.nib_mask, a.nib_magic, a0);
    decode_word_offset136(half ? q.w : q.y, a.nib_mask, a.nib_magic, a1);
#pragma unroll
    for (int j = 0; j < 4; ++j) {   // (q + 136) - 136: exact
      asm("add.rn.bf16x2 %0, %0, %1;" : "+r"(a0[j]) : "r"(a.neg136));
      asm("add.rn.bf16x2 %0, %0, %1;" : "+r"(a1[j]) : "r"(a.neg136));
    }
    const uint32_t sw = half ? sc.y : sc.x;
    const float s_lo = bf16lo_to_f32(sw), s_hi = bf16hi_to_f32(sw);
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      const float zero4[4] = {0.f, 0.f, 0.f, 0.f};
      float c[4];
      mma_bf16_16816(c, a0, bf[n][0], bf[n][1], zero4);
      mma_bf16_16816(c, a1, bf[n][2], bf[n][3], c);
      acc[n][0] = fmaf(s_lo, c[0], acc[n][0]);
      acc[n][1] = fmaf(s_lo, c[1], acc[n][1]);
      acc[n][2] = fmaf(s_hi, c[2], acc[n][2]);
      acc[n][3] = fmaf(s_hi, c[3], acc[n][3]);
    }
  }
}

// One stage of an item of NTL weight tiles of NU units each (K = 64 NU <=
// 512): straight-line code, so the loads and MMAs of all the tiles' units
// interleave (the run-time loops it replaces left TP8's K = 256 down GEMM
// waiting on each unit's loads: 72.9 -> 67.9 us).  Only K = 256 at one
// token tile per pass, outside the SiLU*mul kernels, takes it: compiled into
// those (or a second form for K = 128) it raised their register spills.
template <int NU, int NTL, int NT>
__device__ __forceinline__ void multi_tile_stage(uint32_t st, uint32_t x_off, uint32_t q_off, uint32_t s_off,
                                                 const SmallArgs& a, float (&acc)[NTL][NT][4]) {
#pragma unroll
  for (int t = 0; t < NTL; ++t)
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[t][n][i] = 0.f;
#pragma unroll
  for (int u = 0; u < NU; ++u)
#pragma unroll
    for (int t = 0; t < NTL; ++t)
      unit_mma<NT>(st + (t * NU + u) * kUnitBytes, st + x_off + u * kUnitK * 2, q_off, s_off, a, acc[t]);
}

template <int NT, int STAGES, bool GATHER, int EPI>
__global__ void __launch_bounds__(kThreads, NT == 1 ? 4 : (NT == 2 ? 3 : 2)) gemm_small_kernel(SmallArgs a) {
  using Cfg = SmallCfg<NT>;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full_bar[STAGES];
  __shared__ __align__(8) uint64_t empty_bar[STAGES];
  __shared__ __align__(8) uint64_t item_full[kItemSlots];
  __shared__ __align__(8) uint64_t item_empty[kItemSlots];
  __shared__ SItem item_q[kItemSlots];
  __shared__ int hdr_ok;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    hdr_ok = header_ok(a);
    if (!hdr_ok) set_status(a.status, CHORD_ERR_PREPACK_MISMATCH);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], kConsumerWarps);
    }
    for (int q = 0; q < kItemSlots; ++q) {
      mbar_init(&item_full[q], 1);
      mbar_init(&item_empty[q], kConsumerWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();
  if (!hdr_ok) {
    // A mismatched blob computes nothing (the error is recorded above), but a
    // programmatic launch still waits for the kernel before it and releases
    // the next one only then, so the launch chain keeps its ordering.
    if (a.pdl) {
      grid_dep_wait();
      grid_dep_launch();
    }
    return;
  }

  const int n_units = a.K / kUnitK;
  const int k_stages = (n_units + kUnitsPerStage - 1) / kUnitsPerStage;
  // Short K (one stage per tile): an item covers as many consecutive weight
  // tiles as fill a stage (2 at K = 256, 4 at K = 128), so each mbarrier
  // hand-off carries a full stage of weights and the block's activation
  // rows are loaded once for all of them.
  const int tpi = k_stages == 1 ? max(1, kUnitsPerStage / n_units) : 1;
  const int n_groups = (a.n_tiles + tpi - 1) / tpi;

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    // Items (tile, row block), block index fastest, are taken from a global
    // counter; each is pushed to the consumers through a small ring and its
    // stages are streamed into the shared ring.  The last CTA to run out of
    // items zeroes the counters for the next launch.
    //
    // Programmatic launch: mode 1 waits for the previous kernel before
    // anything else.  Mode 2 reads the expert map and issues the weight
    // copies of the first stages before the wait (weights are never written
    // by the kernels of a layer, and the expert map is complete at launch);
    // the activation rows, the previous kernel's output, follow the wait.
    // The consumers read global memory only through these copies.
    //
    // Item i -> (tile, expert, first sorted row, rows); rows = -1 past the
    // end, 0 for a block whose expert id is out of range (recorded).
    // Loads of the expert map: through the read-only cache in an ordinary
    // launch; in a programmatic one, ordered loads (see grid_dep_wait), from
    // L2 only before the wait.
    auto ld_map = [&](const int32_t* p, int how) {
      return how == 0 ? __ldg(p) : how == 1 ? ld_ca(p) : ld_cg(p);
    };
    const int how = a.pdl ? 1 : 0;   // after the wait
    // item i -> split sp of base item (tile group, block), block index fastest
    auto decode_item = [&](int i, long long total, int nblocks, const SplitPlan& pl, int how) {
      SItem item{0, 0, 0, -1, 1, 0, 0, 0, 0};
      if (i >= 0 && i < total) {   // below zero: counters never zeroed; no item
        int base, sp, ns, slot;
        if (pl.all > 1) {
          base = i / pl.all;
          sp = i - base * pl.all;
          ns = pl.all;
          slot = base;
        } else if (i < pl.head) {
          base = i;
          sp = 0;
          ns = 1;
          slot = 0;
        } else {
          const int j = i - static_cast<int>(pl.head);
          slot = j / pl.tail;
          sp = j - slot * pl.tail;
          ns = pl.tail;
          base = static_cast<int>(pl.head) + slot;
        }
        const int ng = base / nblocks, b = base - ng * nblocks;
        const int e = ld_map(a.expert_ids + b, how);
        item = SItem{ng * tpi, 0, 0, 0, min(tpi, a.n_tiles - ng * tpi), sp * k_stages / ns,
                     (sp + 1) * k_stages / ns, slot, sp | (ns << 16)};
        if (e >= 0 && e < a.E_local) {
          const int row0 = b * a.block_m;
          const int end = ld_map(a.offsets + e, how) + ld_map(a.counts + e, how);
          item.e = e;
          item.row0 = row0;
          item.rows = max(min(a.block_m, end - row0), 0);
        } else {
          set_status(a.status, CHORD_ERR_ROUTING_INVALID);
        }
      }
      return item;
    };
    auto weight_tile = [&](const SItem& item) {
      return a.packed + kPackHeaderBytes +
             (static_cast<size_t>(item.e) * a.n_tiles + item.tile) * static_cast<size_t>(a.tile_bytes);
    };
    // weights of stage ks into ring slot s, the slot expecting `rows` rows too
    // weights of stage ks into ring slot s, the slot expecting `rows` rows
    // too; an item of ntl > 1 tiles (one stage each) copies all of them
    auto issue_weights = [&](const uint8_t* wtile, int ntl, int rows, int ks, int s) {
      const int units = min(kUnitsPerStage, n_units - ks * kUnitsPerStage);
      if (lane == 0) {
        mbar_arrive_expect_tx(&full_bar[s], ntl * units * kUnitBytes + rows * units * kUnitK * 2);
        bulk_g2s(smem + s * Cfg::kStageBytes, wtile + static_cast<size_t>(ks) * kUnitsPerStage * kUnitBytes,
                 ntl * units * kUnitBytes, &full_bar[s]);
      }
      __syncwarp();
    };
    // activation rows of stage ks of one pass into ring slot s
    auto issue_rows = [&](const SItem& item, int pass, int rows, int ks, int s) {
      const int units = min(kUnitsPerStage, n_units - ks * kUnitsPerStage);
      const uint32_t xbytes = units * kUnitK * 2;
      uint8_t* st = smem + s * Cfg::kStageBytes;
      for (int j = lane; j < rows; j += 32) {
        const int r = item.row0 + pass * Cfg::kRowsPerPass + j;
        const int row = GATHER ? ld_map(a.sorted + r, how) / a.topk : r;
        const uint16_t* src = a.A + static_cast<size_t>(row) * a.K + ks * kUnitsPerStage * kUnitK;
        bulk_g2s(st + Cfg::kWBytes + j * kXPitch, src, xbytes, &full_bar[s]);
      }
    };
    int nblocks = 0;
    SItem first{0, 0, 0, -1, 1, 0, 0, 0, 0};
    int pre = 0;   // stages of the first item's first pass already issued
    int i_early = -1;   // mode 1: the first item number, taken before the wait
    if (a.pdl == 2) {
      // The expert map is read from L2 here, never from a copy an SM cached
      // before it was written.
      nblocks = ld_cg(a.ntpp) / a.block_m;
    } else {
      if (a.pdl) {
        // The work counter was cleared before the kernel this one waits for
        // started, so the first item number is claimed now and its round
        // trip overlaps the wait; the item is decoded after it.
        if (lane == 0 && !a.test_timeout) i_early = atomicAdd(a.work, 1);
        i_early = __shfl_sync(0xffffffffu, i_early, 0);
        grid_dep_wait();
        grid_dep_launch();
      }
      nblocks = ld_map(a.ntpp, how) / a.block_m;
    }
    if (nblocks > a.max_blocks || nblocks < 0) {
      set_status(a.status, CHORD_ERR_INVALID_ARG);
      nblocks = nblocks < 0 ? 0 : a.max_blocks;
    }
    // split-K needs one pass per item, a split workspace and more than one
    // stage.  At most half as many items as CTAs: every item splits.  Else,
    // when the last wave holds r = n mod CTAs > CTAs / 2 items, those split
    // into S ranges of at least two stages (S <= kMaxSplit, the partial
    // slots), S giving the shortest last wave if shorter than one item:
    // ceil(r S / CTAs) rounds of ceil(stages / S) stages, each range costing
    // about half a stage more (its partials' round trip).  Measured on GB300:
    // TP8 decode gate/up (r ~ 0.6 of the CTAs, S = 3 or 5) 108.2 -> 106.4 us;
    // below half a wave (EP8 decode gate/up, r ~ 0.3-0.4) or with one-stage
    // ranges (EP8 down, S = 4) splitting was slower (76.6 -> 77.3 us,
    // 43.3 -> 45.5 us): CTAs of a thin last wave share their SMs with few
    // others and finish early anyway.
    const long long n_base = static_cast<long long>(n_groups) * nblocks;
    const long long ctas = gridDim.x;
    SplitPlan plan{1, 1, n_base};
    if (a.partial && a.block_m <= Cfg::kRowsPerPass && k_stages > 1 && n_base > 0) {
      if (2 * n_base <= ctas) {
        int nsplit = static_cast<int>(min(ctas / n_base, static_cast<long long>(min(k_stages, kMaxSplit))));
        nsplit = static_cast<int>(min(static_cast<long long>(nsplit), kSplitSlots / n_base));
        plan.all = nsplit < 2 ? 1 : nsplit;
      } else {
        const long long r = n_base % ctas;
        if (2 * r > ctas && r <= kSplitSlots) {
          long long best = 2LL * k_stages;   // the last wave in half stages, unsplit
          for (int S = 2; S <= min(k_stages / 2, kMaxSplit) && r * S <= Cfg::kSlots; ++S) {
            const long long len = (r * S + ctas - 1) / ctas * (2LL * ((k_stages + S - 1) / S) + 1);
            if (len < best) {
              best = len;
              plan.tail = S;
            }
          }
          if (plan.tail > 1) plan.head = n_base - r;
        }
      }
    }
    const long long total = plan.all > 1 ? n_base * plan.all : plan.head + (n_base - plan.head) * plan.tail;
    if (a.pdl == 2) {
      int i = 0;
      if (lane == 0 && !a.test_timeout) i = atomicAdd(a.work, 1);
      i = __shfl_sync(0xffffffffu, i, 0);
      first = decode_item(a.test_timeout ? static_cast<int>(total) : i, total, nblocks, plan, 2);
      const int rows0 = min(Cfg::kRowsPerPass, first.rows);
      if (rows0 > 0) {
        pre = min(STAGES, first.ks1 - first.ks0);
        for (int j = 0; j < pre; ++j) issue_weights(weight_tile(first), first.ntl, rows0, first.ks0 + j, j);
      }
      grid_dep_wait();
      grid_dep_launch();
      for (int j = 0; j < pre; ++j) issue_rows(first, 0, rows0, first.ks0 + j, j);
    }
    int it = 0, q = 0;
    bool ok = !a.test_timeout, use_first = a.pdl == 2 && !a.test_timeout;   // test hook: no item at all
    // Items of one K stage are short next to the round trips of the counter
    // and the expert map, so they are taken two at a time: lane j decodes
    // item base + j, and the loop hands them out in order (TP8 down GEMM
    // 73.8 -> 72.2 us; four or eight at a time measured no better or worse).
    const int batch = (k_stages + plan.all - 1) / plan.all <= 1 ? 2 : 1;
    SItem held{0, 0, 0, -1, 1, 0, 0, 0, 0};
    int held_k = 0, held_n = 0;
    while (ok) {
      SItem item;
      if (use_first) {   // fetched before the wait
        item = first;
        use_first = false;
      } else {
        if (held_k == held_n) {
          int i = 0, nb = batch;
          if (i_early >= 0) {
            i = i_early;
            nb = 1;
            i_early = -1;
          } else {
            if (lane == 0) i = atomicAdd(a.work, batch);
            i = __shfl_sync(0xffffffffu, i, 0);
          }
          held = decode_item(lane < nb ? i + lane : static_cast<int>(total), total, nblocks, plan, how);
          held_k = 0;
          held_n = nb;
        }
        item.tile = __shfl_sync(0xffffffffu, held.tile, held_k);
        item.e = __shfl_sync(0xffffffffu, held.e, held_k);
        item.row0 = __shfl_sync(0xffffffffu, held.row0, held_k);
        item.rows = __shfl_sync(0xffffffffu, held.rows, held_k);
        item.ntl = __shfl_sync(0xffffffffu, held.ntl, held_k);
        item.ks0 = __shfl_sync(0xffffffffu, held.ks0, held_k);
        item.ks1 = __shfl_sync(0xffffffffu, held.ks1, held_k);
        item.slot = __shfl_sync(0xffffffffu, held.slot, held_k);
        item.split = __shfl_sync(0xffffffffu, held.split, held_k);
        ++held_k;
      }
      const int slot = q % kItemSlots;
      if (q >= kItemSlots)
        ok = mbar_wait_backoff(&item_empty[slot], ((q / kItemSlots) - 1) & 1, a.status, a.wait_polls);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      if (lane == 0) {
        item_q[slot] = item;
        mbar_arrive(&item_full[slot]);
      }
      ++q;
      if (item.rows < 0) break;
      const uint8_t* wtile = weight_tile(item);
      const int passes = (item.rows + Cfg::kRowsPerPass - 1) / Cfg::kRowsPerPass;
      for (int pass = 0; pass < passes && ok; ++pass) {
        const int rows = min(Cfg::kRowsPerPass, item.rows - pass * Cfg::kRowsPerPass);
        for (int ks = item.ks0; ks < item.ks1; ++ks, ++it) {
          if (pre > 0) {   // issued before the wait (first pass of the first item: it == ks - ks0)
            --pre;
            continue;
          }
          const int s = it % STAGES;
          if (it >= STAGES) ok = mbar_wait_backoff(&empty_bar[s], ((it / STAGES) - 1) & 1, a.status, a.wait_polls);
          ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
          if (!ok) break;
          issue_weights(wtile, item.ntl, rows, ks, s);
          issue_rows(item, pass, rows, ks, s);
        }
      }
    }
    if (lane == 0) {
      // every CTA arrives, also one that gave up on a wait, so the counters
      // are zero again after the launch whatever happened
      if (atomicAdd(a.work + 1, 1) == static_cast<int>(gridDim.x) - 1) {
        atomicExch(a.work, 0);
        atomicExch(a.work + 1, 0);
      }
      // Before leaving, make sure no copy into this CTA's smem is in flight.
      for (int j = max(0, it - STAGES); j < it; ++j)
        mbar_wait(&full_bar[j % STAGES], (j / STAGES) & 1, a.status);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int g = lane >> 2, t = lane & 3;
  const uint32_t smem_base = smem_u32(smem);
  const uint32_t q_off = warp * 512 + lane * 16;             // this warp's slab, this lane
  const uint32_t s_off = kUnitQBytes + warp * 64 + g * 8;
  const uint32_t x_off = Cfg::kWBytes + (lane & 7) * kXPitch + (lane >> 3) * 16;
  int it = 0;
  for (int q = 0;; ++q) {
    const int slot = q % kItemSlots;
    if (!mbar_wait(&item_full[slot], (q / kItemSlots) & 1, a.status, a.wait_polls)) return;
    const SItem item = item_q[slot];
    __syncwarp();
    if (lane == 0) mbar_arrive(&item_empty[slot]);
    if (item.rows < 0) return;
    const int passes = (item.rows + Cfg::kRowsPerPass - 1) / Cfg::kRowsPerPass;
    const int sp = item.split & 0xffff, nsplit = item.split >> 16;
    // BF16 output of one 64-row weight tile for `rows` token rows from r0
    auto epilogue = [&](int tile, const float (&acc)[NT][4], int rows, size_t r0) {
#pragma unroll
      for (int n = 0; n < NT; ++n) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int tok = n * 8 + 2 * t + i;
          if (tok >= rows) continue;
          if (EPI == CHORD_EPI_WEIGHTED_ADD) {
            // the row's assignment f: token f / topk, weight topk_w[f]
            // (read from L2: written by earlier kernels); padding rows skip
            const int f = ld_cg(a.sorted + r0 + tok);
            if (f < 0 || f >= a.M * a.topk) continue;
            const float w = ld_cg(a.topk_w + f);
            float* crow = a.Cf + static_cast<size_t>(f / a.topk) * a.N;
            const int col = kTileRows * tile + 16 * warp + g;
            if (col < a.N) atomicAdd(crow + col, w * acc[n][i]);
            if (col + 8 < a.N) atomicAdd(crow + col + 8, w * acc[n][2 + i]);
            continue;
          }
          uint16_t* crow = a.C + (r0 + tok) * a.ldc;
          if (EPI == CHORD_EPI_SILU_MUL) {
            // acc[n][i]: gate of index i0 + g; acc[n][2 + i]: up of the same index
            const int col = 32 * tile + 8 * warp + g;
            crow[col] = f32_to_bf16_rn(silu_f32(acc[n][i]) * acc[n][2 + i]);
          } else {
            const int col = kTileRows * tile + 16 * warp + g;
            if (col < a.N) crow[col] = f32_to_bf16_rn(acc[n][i]);
            if (col + 8 < a.N) crow[col + 8] = f32_to_bf16_rn(acc[n][2 + i]);
          }
        }
      }
    };
    if (item.ntl > 1) {
      // several tiles, one stage (K <= 512): per pass, tile by tile
      for (int pass = 0; pass < passes; ++pass, ++it) {
        const int rows = min(Cfg::kRowsPerPass, item.rows - pass * Cfg::kRowsPerPass);
        const int s = it % STAGES;
        if (!mbar_wait(&full_bar[s], (it / STAGES) & 1, a.status, a.wait_polls)) return;
        const uint32_t st = smem_base + s * Cfg::kStageBytes;
        const size_t r0 = static_cast<size_t>(item.row0) + pass * Cfg::kRowsPerPass;
        if (NT == 1 && EPI != CHORD_EPI_SILU_MUL && n_units == 4 && item.ntl == 2) {   // K = 256 (down GEMMs)
          float acc[2][NT][4];
          multi_tile_stage<4, 2, NT>(st, x_off, q_off, s_off, a, acc);
          epilogue(item.tile, acc[0], rows, r0);
          epilogue(item.tile + 1, acc[1], rows, r0);
        } else
#pragma unroll 1
        for (int tl = 0; tl < item.ntl; ++tl) {
          float acc[NT][4];
#pragma unroll
          for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[n][i] = 0.f;
#pragma unroll 1
          for (int u = 0; u < n_units; ++u)
            unit_mma<NT>(st + (tl * n_units + u) * kUnitBytes, st + x_off + u * kUnitK * 2, q_off, s_off, a, acc);
          epilogue(item.tile + tl, acc, rows, static_cast<size_t>(item.row0) + pass * Cfg::kRowsPerPass);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[s]);
      }
      continue;
    }
    for (int pass = 0; pass < passes; ++pass) {
      const int rows = min(Cfg::kRowsPerPass, item.rows - pass * Cfg::kRowsPerPass);
      float acc[NT][4];
#pragma unroll
      for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[n][i] = 0.f;

      for (int ks = item.ks0; ks < item.ks1; ++ks, ++it) {
        const int s = it % STAGES;
        if (!mbar_wait(&full_bar[s], (it / STAGES) & 1, a.status, a.wait_polls)) return;
        const uint32_t st = smem_base + s * Cfg::kStageBytes;
        const int units = min(kUnitsPerStage, n_units - ks * kUnitsPerStage);
        if (units == kUnitsPerStage) {
#pragma unroll
          for (int u = 0; u < kUnitsPerStage; ++u)
            unit_mma<NT>(st + u * kUnitBytes, st + x_off + u * kUnitK * 2, q_off, s_off, a, acc);
        } else {
#pragma unroll 1
          for (int u = 0; u < units; ++u)
            unit_mma<NT>(st + u * kUnitBytes, st + x_off + u * kUnitK * 2, q_off, s_off, a, acc);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[s]);
      }

      if (nsplit > 1) {
        // split-K (one pass per item): publish this split's partial, and
        // the last split of the item to arrive adds all of them in split
        // order and runs the epilogue
        float* slot_base = a.partial + static_cast<size_t>(item.slot) * nsplit * Cfg::kSlotFloats;
        float4* mine = reinterpret_cast<float4*>(slot_base + static_cast<size_t>(sp) * Cfg::kSlotFloats +
                                                 (warp * 32 + lane) * 4 * NT);
#pragma unroll
        for (int n = 0; n < NT; ++n) mine[n] = make_float4(acc[n][0], acc[n][1], acc[n][2], acc[n][3]);
        __threadfence();
        __syncwarp();
        int prev = 0;
        if (lane == 0) prev = atomicAdd(a.split_cnt + item.slot * kConsumerWarps + warp, 1);
        prev = __shfl_sync(0xffffffffu, prev, 0);
        if (prev != nsplit - 1) continue;   // not the last split of this item
        __threadfence();
        if (lane == 0) atomicExch(a.split_cnt + item.slot * kConsumerWarps + warp, 0);   // ready for the next launch
        float sum[NT][4];
        for (int k = 0; k < nsplit; ++k) {
#pragma unroll
          for (int n = 0; n < NT; ++n) {
            float4 v;
            if (k == sp) {
              v = make_float4(acc[n][0], acc[n][1], acc[n][2], acc[n][3]);
            } else {
              v = ld_cg_f4(slot_base + static_cast<size_t>(k) * Cfg::kSlotFloats + (warp * 32 + lane) * 4 * NT + 4 * n);
            }
            if (k == 0) {
              sum[n][0] = v.x; sum[n][1] = v.y; sum[n][2] = v.z; sum[n][3] = v.w;
            } else {
              sum[n][0] += v.x; sum[n][1] += v.y; sum[n][2] += v.z; sum[n][3] += v.w;
            }
          }
        }
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
          for (int i = 0; i < 4; ++i) acc[n][i] = sum[n][i];
      }

      epilogue(item.tile, acc, rows, static_cast<size_t>(item.row0) + pass * Cfg::kRowsPerPass);
    }
  }
}

template <int NT, int STAGES, bool GATHER, int EPI>
cudaError_t launch_small(const SmallArgs& a, cudaStream_t st) {
  const int smem = STAGES * SmallCfg<NT>::kStageBytes;
  auto kern = gemm_small_kernel<NT, STAGES, GATHER, EPI>;
  cudaError_t err = ensure_smem_limit<gemm_small_kernel<NT, STAGES, GATHER, EPI>>(smem);
  if (err != cudaSuccess) return err;
  static int per_sm[64] = {0}, sms[64] = {0};
  int dev = 0;
  err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!per_sm[dev]) {
    int n = 0, m = 0;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kThreads, smem);
    if (err != cudaSuccess) return err;
    err = cudaDeviceGetAttribute(&m, cudaDevAttrMultiProcessorCount, dev);
    if (err != cudaSuccess) return err;
    sms[dev] = m;
    per_sm[dev] = n > 0 ? n : 1;
  }
  return launch_kernel(kern, dim3(per_sm[dev] * sms[dev]), dim3(kThreads), smem, st, a.pdl != 0, a);
}

template <int NT, int STAGES>
cudaError_t dispatch_mode(const SmallArgs& a, bool gather, int epi, cudaStream_t st) {
  if (gather) {
    if (epi == CHORD_EPI_WEIGHTED_ADD) return cudaErrorInvalidValue;   // refused by the host checks
    return epi == CHORD_EPI_SILU_MUL ? launch_small<NT, STAGES, true, CHORD_EPI_SILU_MUL>(a, st)
                                     : launch_small<NT, STAGES, true, CHORD_EPI_STORE>(a, st);
  }
  if (epi == CHORD_EPI_WEIGHTED_ADD) return launch_small<NT, STAGES, false, CHORD_EPI_WEIGHTED_ADD>(a, st);
  return epi == CHORD_EPI_SILU_MUL ? launch_small<NT, STAGES, false, CHORD_EPI_SILU_MUL>(a, st)
                                   : launch_small<NT, STAGES, false, CHORD_EPI_STORE>(a, st);
}

}  // namespace

cudaError_t gemm_small_launch(const GemmLaunch& g, int rows_per_pass, cudaStream_t st) {
  SmallArgs a;
  a.A = g.A;
  a.packed = static_cast<const uint8_t*>(g.packed);
  a.sorted = g.sorted;
  a.expert_ids = g.expert_ids;
  a.ntpp = g.ntpp;
  a.counts = g.counts;
  a.offsets = g.offsets;
  a.work = g.work;
  a.block_m = g.block_m;
  a.C = g.C;
  a.status = g.status;
  a.N = g.N;
  a.K = g.K;
  a.M = g.M;
  a.topk = g.topk;
  a.Cf = g.Cf;
  a.topk_w = g.topk_w;
  a.E_local = g.E_local;
  a.pdl = g.pdl;
  a.max_blocks = g.max_blocks;
  a.partial = g.split_cnt ? g.split_partial : nullptr;
  a.test_timeout = g.test_timeout;
  a.wait_polls = g.test_timeout ? kTestWaitPolls : kWaitPolls;
  a.split_cnt = g.split_cnt;
  const PackHeader h = make_pack_header(g.E_local, g.N, g.K, g.epilogue == CHORD_EPI_SILU_MUL);
  a.n_tiles = h.n_tiles;
  a.tile_bytes = h.tile_bytes;
  a.need_flags = g.epilogue == CHORD_EPI_SILU_MUL ? kPackFlagGateUp : 0u;
  a.ldc = g.epilogue == CHORD_EPI_SILU_MUL ? g.N / 2 : g.N;
  a.nib_mask = 0x000F000Fu;
  a.nib_magic = 0x43004300u;
  a.neg136 = kBf16x2Neg136;
  // 2 stages: 53.5 KB (NT=1, 4 CTAs/SM), 70.2 KB (NT=2, 3 CTAs/SM), 103.5 KB (NT=4, 2 CTAs/SM)
  if (rows_per_pass <= 8) return dispatch_mode<1, 2>(a, g.gather, g.epilogue, st);
  if (rows_per_pass <= 16) return dispatch_mode<2, 2>(a, g.gather, g.epilogue, st);
  return dispatch_mode<4, 2>(a, g.gather, g.epilogue, st);
}

}  // namespace chord
