// Large-M (prefill) indexed W4A16 MoE GEMM on the 5th-generation tensor cores.
//
// [Humming] "워크로드별 튜닝 및 JIT 컴파일": at larger batch a TMA + UMMA
// pipeline gives the better throughput; [Chord] "그룹 SM90 커널 기법": a
// persistent warp-specialised main loop pipelining TMA loads, dequantisation
// and the MMA.  Design on sm_103a (one CTA per SM, persistent):
//   * work item = (local expert, 128 weight rows, pass of up to 192 of the
//     expert's rows), numbered expert by expert; warp 0 takes the next
//     number from a global counter (items differ in rows, so a static deal
//     leaves SMs idle), decodes it and hands it to the other roles through
//     a small mbarrier ring; the CTAs running at one time cover a few experts, whose
//     activation rows stay in L2; the last CTA to run dry zeroes the counter;
//   * the MMA is "swap AB": the 128 weight rows are M, the expert's rows
//     (tokens) are N (a multiple of 16 up to 192), so an expert's rows are
//     padded to 16, not to 128;
//   * the dequantised weights (A) never touch shared memory: the dequant
//     warps write them into tensor memory with tcgen05.st (the packed
//     fragment order is the 16x128b store order) and tcgen05.mma reads A
//     from TMEM; only the activations (B) are read from shared memory, which
//     halves the shared-memory traffic per MMA;
//   * one pipeline stage is 128 of K (eight K=16 MMAs), so every mbarrier
//     handshake covers twice the tensor work of a 64-wide stage;
//   * three rings, each with its own full/empty mbarriers: packed weights
//     (shared memory, 6 deep, from HBM, 1-D bulk copies by warp 0),
//     activation tiles (shared memory, 3 deep, from L2, one 2-D TMA box of
//     up to 192 rows per 64 of K, 128-byte swizzle, by warp 2) and
//     dequantised A tiles (TMEM, 2 deep);
//   * warps 4-19 (dequant): two groups of eight take alternate stages (each
//     group owns one A slot); in a group, each warp covers one 32-row TMEM
//     lane quarter and one 64-wide half of the stage: INT4 -> BF16 q*s
//     (rounded once), tcgen05.st.  A warp's stage is a chain of latencies
//     (barrier waits, shared-memory loads, decode, TMEM store and fences,
//     ~1.3k cycles measured), longer than the stage's MMAs, so one group
//     alone left the tensor pipe idle; two groups halve the gap (prefill
//     gate/up 593 -> 536 us on GB300); the waits on two barriers probe both
//     at once (one probe latency instead of two: 531 -> 511 us);
//   * warp 1 (MMA): TMEM allocation; the converged warp waits and one
//     elected lane issues the MMAs (M=128) into one of two accumulators and
//     commits slot release and item completion to mbarriers;
//   * warps 20-23 (epilogue): tcgen05.ld of the accumulator, SiLU(gate) * up
//     (gate and up rows of one index sit 8 TMEM lanes apart) or a plain
//     store, BF16, rows in sorted order; the second accumulator lets the next
//     item's MMAs run meanwhile.
// TMEM: accumulators at columns 0 and 192, A slots at 384 and 448.
// Every mbarrier wait is bounded; on a timeout the CTA records
// CHORD_ERR_TIMEOUT, drains its own copies and MMAs, frees TMEM and exits.
#include "common.cuh"
#include "kernels.h"
#include "tc5.cuh"

namespace chord {
namespace {

constexpr int kMRows = 128;                      // weight rows per item (2 packed tiles)
constexpr int kMaxTok = 192;                     // tokens per pass (MMA N)
constexpr int kAccBufs = 2;                      // TMEM accumulators: the epilogue overlaps the next item
constexpr int kStageUnits = 2;                   // 64-wide K units per stage
constexpr int kSP = 6, kSB = 3, kSA = 2;         // ring depths: packed, activations, A in TMEM
constexpr int kBHalfBytes = kMaxTok * kUnitK * 2;            // 24 KB: 192 rows x 128 B
constexpr int kBStageBytes = kStageUnits * kBHalfBytes;      // 48 KB
constexpr int kPStageBytes = 2 * kStageUnits * kUnitBytes;   // 9216: [tile][unit]
constexpr int kBOff = 0, kPOff = kSB * kBStageBytes;
constexpr int kSmemBytes = kPOff + kSP * kPStageBytes + 1024;   // + alignment slack
constexpr int kAccCols = kMaxTok;                // accumulator j at column j * kMaxTok
constexpr int kACol0 = kAccBufs * kAccCols;      // A slot s at column kACol0 + 64 s
constexpr int kASlotCols = kStageUnits * kUnitK / 2;         // 64
constexpr int kTmemCols = 512;
static_assert(kACol0 + kSA * kASlotCols <= kTmemCols, "TMEM budget");
static_assert(kMaxTok % 64 == 0 && kMaxTok <= 256, "whole 64-row boxes never overrun an activation slot");
// Two groups of eight dequant warps take alternate stages.  With two A
// slots each group owns one slot (stage it uses slot it % 2 and group
// it % 2), so a group waits for exactly the previous phase of its own slot
// and the parity waits cannot alias; a third group would need a third slot.
constexpr int kGroups = 2;
constexpr int kDequantWarp0 = 4, kGroupWarps = 8, kDequantWarps = kGroups * kGroupWarps;
static_assert(kGroups == kSA, "each dequant group owns one A slot");
constexpr int kEpiWarp0 = kDequantWarp0 + kDequantWarps;   // 20: warp index % 4 = lane quarter
constexpr int kThreads = 32 * (kEpiWarp0 + 4);
constexpr int kMaxExperts = 1024;
constexpr int kItemSlots = 4;
// roles that read each item from the ring: activation producer, MMA warp,
// dequant warps, epilogue warps
constexpr int kItemReaders = 1 + 1 + kDequantWarps + 4;
static_assert(kSmemBytes + (kMaxExperts + 1) * 4 + 512 <= 232448, "shared memory budget");
static_assert((kBHalfBytes % 1024) == 0 && (kPOff % 1024) == 0, "SW128 tiles");
static_assert((kDequantWarp0 % 4) == 0 && (kEpiWarp0 % 4) == 0, "warp index selects the TMEM lane quarter");

struct LargeArgs {
  const uint8_t* packed;
  const int32_t* counts;
  const int32_t* offsets;
  int* work;        // [0] next item, [1] CTAs done; zero before the launch, zero after it
  uint16_t* C;
  float* Cf;             // weighted add: FP32 [M, N] accumulator (else NULL)
  const float* topk_w;   // weighted add: routing weights [M, topk]
  const int32_t* sorted; // weighted add: sorted_token_ids
  int M, topk;
  int* status;
  int N, K, ldc, E_local, n_blob_tiles;
  int64_t tile_bytes;
  uint32_t need_flags;
  int gate_up;
  int box_s, box_b;               // activation box heights (rows): small items / the rest
  uint32_t nib_mask, nib_magic;   // decode constants, passed at run time so they stay in registers
};

// tcgen05.mma / commit issued by one elected lane of a converged warp (the
// operands are warp-uniform), which keeps the issue path short.
__device__ __forceinline__ void mma_ts_elect(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred q, e;\n\t.reg .b32 r;\n\t"
      "elect.sync r|e, 0xffffffff;\n\t"
      "setp.ne.b32 q, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, q;\n\t}" ::"r"(d),
      "r"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void commit_elect(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t.reg .b32 r;\n\t"
      "elect.sync r|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
          smem_u32(bar))
      : "memory");
}
struct Item {
  int e, wt, row0, rows;
};

__device__ __forceinline__ bool header_ok(const LargeArgs& a) {
  const PackHeader* h = reinterpret_cast<const PackHeader*>(a.packed);
  return h->magic == kPackMagic && h->version == kPackVersion && h->N == a.N && h->K == a.K &&
         h->group == kGroup && h->E >= a.E_local && h->tile_bytes == a.tile_bytes &&
         (h->flags & a.need_flags) == a.need_flags;
}

// Item i of the global list (experts in order; per expert, passes, then
// 128-row weight tiles).  prefix[e] = first item of expert e.
__device__ __forceinline__ Item item_of(int i, const int* prefix, const int32_t* counts,
                                        const int32_t* offsets, int E, int n_wt) {
  int lo = 0, hi = E - 1;  // largest e with prefix[e] <= i
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= i) lo = mid; else hi = mid - 1;
  }
  const int e = lo, cnt = __ldg(counts + e);
  const int local = i - prefix[e];
  const int p = local / n_wt, wt = local - p * n_wt;
  const int n_pass = (cnt + kMaxTok - 1) / kMaxTok;
  const int tp = ((cnt + n_pass - 1) / n_pass + 15) & ~15;
  Item it;
  it.e = e;
  it.wt = wt;
  it.row0 = __ldg(offsets + e) + p * tp;
  it.rows = min(tp, cnt - p * tp);
  return it;
}

// Dequantise this lane's part of two 16-row slabs of one 64-wide K unit
// (packed fragment order) into BF16 q*s pairs, 16 registers per slab in the
// tcgen05.st 16x128b order: per K=16 step j, fragment registers a0..a3.
__device__ __forceinline__ void dequant_two_slabs(const uint8_t* pst, const uint32_t (&q_off)[2],
                                                  const uint32_t (&s_off)[2], uint32_t mask, uint32_t magic,
                                                  uint32_t (&v)[2][16]) {
  const __nv_bfloat162 k136 = __floats2bfloat162_rn(136.f, 136.f);
#pragma unroll
  for (int sl = 0; sl < 2; ++sl) {
    const uint4 qw = *reinterpret_cast<const uint4*>(pst + q_off[sl]);
    const uint2 sc = *reinterpret_cast<const uint2*>(pst + s_off[sl]);
    const uint32_t w4[4] = {qw.x, qw.y, qw.z, qw.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {   // K=16 step j; scale group j / 2
      const uint32_t sw = (j >> 1) ? sc.y : sc.x;
      const uint32_t s_lo = __byte_perm(sw, sw, 0x1010);   // {s[g], s[g]}
      const uint32_t s_hi = __byte_perm(sw, sw, 0x3232);   // {s[g+8], s[g+8]}
      uint32_t d[4];
      decode_word_offset136(w4[j], mask, magic, d);
#pragma unroll
      for (int r = 0; r < 4; ++r) {   // d[r]: fragment register a_r (rows g, g+8, g, g+8)
        __nv_bfloat162 x = *reinterpret_cast<__nv_bfloat162*>(&d[r]);
        x = __hsub2(x, k136);
        const uint32_t sr = (r & 1) ? s_hi : s_lo;
        x = __hmul2(x, *reinterpret_cast<const __nv_bfloat162*>(&sr));
        v[sl][4 * j + r] = *reinterpret_cast<uint32_t*>(&x);
      }
    }
  }
}

// Next item from the CTA's item ring (consumer q of this role): the global
// item number, -1 at the end of the work, -2 on a timeout, and in *out (when
// given) the item as the producer decoded it, read before the slot is
// released.  All lanes of the calling warp wait; lane 0 releases the slot.
__device__ __forceinline__ int take_item(uint64_t* item_full, uint64_t* item_empty, const volatile int* item_q,
                                         const volatile int (*item_f)[kItemSlots], int q, int* status,
                                         Item* out) {
  const int slot = q % kItemSlots;
  if (!mbar_wait(&item_full[slot], (q / kItemSlots) & 1, status)) return -2;
  const int i = item_q[slot];
  if (out) {
    out->e = item_f[0][slot];
    out->wt = item_f[1][slot];
    out->row0 = item_f[2][slot];
    out->rows = item_f[3][slot];
  }
  __syncwarp(__activemask());
  if ((threadIdx.x & 31) == 0) mbar_arrive(&item_empty[slot]);
  return i;
}

// 64-wide K units in stage ks (the last stage of a K that is an odd number
// of units holds one).
__device__ __forceinline__ int stage_units(int ks, int n_units) {
  return min(kStageUnits, n_units - ks * kStageUnits);
}

__global__ void __launch_bounds__(kThreads, 1)
    gemm_large_kernel(const __grid_constant__ CUtensorMap map_s, const __grid_constant__ CUtensorMap map_b,
                      LargeArgs a) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t p_full[kSP], p_empty[kSP];
  __shared__ __align__(8) uint64_t b_full[kSB], b_empty[kSB];
  __shared__ __align__(8) uint64_t a_full[kSA], a_empty[kSA];
  __shared__ __align__(8) uint64_t tfull_bar[kAccBufs], tempty_bar[kAccBufs], done_bar;
  __shared__ __align__(8) uint64_t item_full[kItemSlots], item_empty[kItemSlots];
  __shared__ volatile int item_q[kItemSlots];
  __shared__ volatile int item_f[4][kItemSlots];   // the item's e, wt, row0, rows
  __shared__ uint32_t tmem_base_s;
  __shared__ int prefix[kMaxExperts + 1];
  __shared__ int hdr_ok;
  __shared__ volatile int abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t smem0 = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (smem0 - smem_u32(smem_raw));
  const int E = a.E_local;
  const int n_wt = a.N / kMRows;
  const int n_units = a.K / kUnitK;
  const int n_stages = (n_units + kStageUnits - 1) / kStageUnits;

  if (tid == 0) {
    hdr_ok = header_ok(a);
    if (!hdr_ok) set_status(a.status, CHORD_ERR_PREPACK_MISMATCH);
    abort_flag = 0;
    for (int s = 0; s < kSP; ++s) {
      mbar_init(&p_full[s], 1);
      mbar_init(&p_empty[s], kGroupWarps);
    }
    for (int s = 0; s < kSB; ++s) {
      mbar_init(&b_full[s], 1);
      mbar_init(&b_empty[s], 1);
    }
    for (int s = 0; s < kSA; ++s) {
      mbar_init(&a_full[s], kGroupWarps);
      mbar_init(&a_empty[s], 1);
    }
    for (int b = 0; b < kAccBufs; ++b) {
      mbar_init(&tfull_bar[b], 1);
      mbar_init(&tempty_bar[b], 4);
    }
    mbar_init(&done_bar, 1);
    for (int q = 0; q < kItemSlots; ++q) {
      mbar_init(&item_full[q], 1);
      mbar_init(&item_empty[q], kItemReaders);
    }
    fence_mbar_init();
  }
  // the item prefix over experts
  if (warp == 0) {
    int run = 0;
    for (int base = 0; base < E; base += 32) {
      const int e = base + lane;
      int items = 0;
      const int cnt = e < E ? __ldg(a.counts + e) : 0;
      if (cnt > 0) items = n_wt * ((cnt + kMaxTok - 1) / kMaxTok);
      int inc = items;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += t;
      }
      if (e < E) prefix[e] = run + inc - items;
      run += __shfl_sync(0xffffffffu, inc, 31);
    }
    if (lane == 0) prefix[E] = run;
  }
  if (warp == 1) tmem_alloc(&tmem_base_s, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = tmem_base_s;
  const int total_items = hdr_ok ? prefix[E] : 0;

  if (warp == 0) {
    // ------------------------------------------------ packed-weight producer
    if (lane == 0) {
      int it = 0;
      for (int q = 0;; ++q) {
        int i = atomicAdd(a.work, 1);
        if (i < 0 || i >= total_items || abort_flag) i = -1;   // below zero: counters never zeroed
        const int slot = q % kItemSlots;
        if (q >= kItemSlots && !mbar_wait_backoff(&item_empty[slot], ((q / kItemSlots) - 1) & 1, a.status)) {
          abort_flag = 1;
          break;
        }
        // the item is decoded once, here, and handed to the other roles with
        // its number (their item_of lookups were global loads on the path
        // from one item to the next)
        Item item{0, 0, 0, 0};
        if (i >= 0) item = item_of(i, prefix, a.counts, a.offsets, E, n_wt);
        item_f[0][slot] = item.e;
        item_f[1][slot] = item.wt;
        item_f[2][slot] = item.row0;
        item_f[3][slot] = item.rows;
        item_q[slot] = i;
        mbar_arrive(&item_full[slot]);   // release: the item is visible to the waiters
        if (i < 0) break;
        const uint8_t* t0 = a.packed + kPackHeaderBytes +
                            (static_cast<size_t>(item.e) * a.n_blob_tiles + 2 * item.wt) *
                                static_cast<size_t>(a.tile_bytes);
        for (int ks = 0; ks < n_stages; ++ks, ++it) {
          const int s = it % kSP;
          if (it >= kSP && !mbar_wait_backoff(&p_empty[s], ((it / kSP) - 1) & 1, a.status)) {
            abort_flag = 1;
            break;
          }
          const uint32_t bytes = stage_units(ks, n_units) * kUnitBytes;
          const size_t src = static_cast<size_t>(ks) * kStageUnits * kUnitBytes;
          uint8_t* dst = smem + kPOff + s * kPStageBytes;
          mbar_arrive_expect_tx(&p_full[s], 2 * bytes);
          bulk_g2s(dst, t0 + src, bytes, &p_full[s]);
          bulk_g2s(dst + kStageUnits * kUnitBytes, t0 + a.tile_bytes + src, bytes, &p_full[s]);
        }
      }
      // the last CTA to run out of items zeroes the counters for the next
      // launch; every CTA arrives, also one that gave up on a wait
      if (atomicAdd(a.work + 1, 1) == static_cast<int>(gridDim.x) - 1) {
        atomicExch(a.work, 0);
        atomicExch(a.work + 1, 0);
      }
      // drain: every issued copy must land before the CTA can exit
      for (int j = max(0, it - kSP); j < it; ++j)
        mbar_wait(&p_full[j % kSP], (j / kSP) & 1, a.status);
    }
  } else if (warp == 2) {
    // ------------------------------------------------- activation producer
    if (lane == 0) {
      int it = 0;
      for (int q = 0; !abort_flag; ++q) {
        Item item;
        const int i = take_item(item_full, item_empty, item_q, item_f, q, a.status, &item);
        if (i < 0) {
          if (i == -2) abort_flag = 1;
          break;
        }
        const int n_mma = (item.rows + 15) & ~15;
        const bool small = n_mma <= a.box_s;
        const CUtensorMap* map = small ? &map_s : &map_b;
        const int box = small ? a.box_s : a.box_b;
        const int nbox = (n_mma + box - 1) / box;   // box divides 192: nbox * box <= 192
        for (int ks = 0; ks < n_stages; ++ks, ++it) {
          const int s = it % kSB;
          if (it >= kSB && !mbar_wait_backoff(&b_empty[s], ((it / kSB) - 1) & 1, a.status)) {
            abort_flag = 1;
            break;
          }
          const int nu = stage_units(ks, n_units);
          uint8_t* dst = smem + kBOff + s * kBStageBytes;
          mbar_arrive_expect_tx(&b_full[s], nu * nbox * box * kUnitK * 2);
          for (int h = 0; h < nu; ++h)
            for (int b = 0; b < nbox; ++b)
              tma_load_2d(dst + h * kBHalfBytes + b * box * kUnitK * 2, map,
                          (ks * kStageUnits + h) * kUnitK, item.row0 + b * box, &b_full[s]);
        }
      }
      for (int j = max(0, it - kSB); j < it; ++j)
        mbar_wait(&b_full[j % kSB], (j / kSB) & 1, a.status);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs this loop (all lanes wait on the same barriers);
    // one elected lane issues each MMA and commit.
    {
      int it = 0, j = 0;
      bool issued_any = false;
      for (; !abort_flag; ++j) {
        Item item;
        int i = take_item(item_full, item_empty, item_q, item_f, j, a.status, &item);
        i = __shfl_sync(0xffffffffu, i, 0);   // warp-uniform before elect.sync
        if (i < 0) {
          if (i == -2) abort_flag = 1;
          break;
        }
        const int acc = j % kAccBufs, use = j / kAccBufs;
        if (use >= 1 && !mbar_wait(&tempty_bar[acc], (use - 1) & 1, a.status)) {
          abort_flag = 1;
          break;
        }
        tc_fence_after();
        const int n_mma = (item.rows + 15) & ~15;
        const uint32_t idesc = idesc_bf16_f32(kMRows, n_mma);
        const uint32_t d_tmem = tmem_base + acc * kAccCols;
        for (int ks = 0; ks < n_stages; ++ks, ++it) {
          const int sa = it % kSA, sb = it % kSB;
          if (!mbar_wait2(&a_full[sa], (it / kSA) & 1, &b_full[sb], (it / kSB) & 1, a.status)) {
            abort_flag = 1;
            break;
          }
          tc_fence_after();
          const uint32_t a_tmem = tmem_base + kACol0 + sa * kASlotCols;
          const uint32_t b_base = smem0 + kBOff + sb * kBStageBytes;
          const uint64_t bd0 = sw128_kmajor_desc(b_base);
          const uint32_t acc0 = ks != 0 ? 1u : 0u;
          if (stage_units(ks, n_units) == kStageUnits) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ts_elect(d_tmem, a_tmem + 8 * kk, bd0 + (kk >> 2) * (kBHalfBytes >> 4) + 2 * (kk & 3), idesc,
                             kk ? 1u : acc0);
          } else {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_ts_elect(d_tmem, a_tmem + 8 * kk, bd0 + 2 * kk, idesc, kk ? 1u : acc0);
          }
          commit_elect(&a_empty[sa]);
          commit_elect(&b_empty[sb]);
          issued_any = true;
        }
        if (abort_flag) break;
        commit_elect(&tfull_bar[acc]);
      }
      // all issued MMAs complete before TMEM can be freed
      if (issued_any) {
        commit_elect(&done_bar);
        mbar_wait(&done_bar, 0, a.status);
      }
    }
  } else if (warp >= kDequantWarp0 && warp < kEpiWarp0) {
    // ------------------------------------------------------------ dequant
    // This warp: TMEM lane quarter q (rows 32q..32q+31 = slabs 2q, 2q+1 of
    // the 128-row item) and unit hu (K 64*hu .. 64*hu+63) of each stage.
    const int dq = warp - kDequantWarp0;
    const int grp = dq / kGroupWarps;
    const int q = warp & 3, hu = (dq % kGroupWarps) >> 2;
    const int g = lane >> 2;
    const uint32_t mask = a.nib_mask, magic = a.nib_magic;   // run-time: kept in registers
    // packed offsets of slab sl (0, 1) within a stage: tile, unit, slab-in-tile
    uint32_t q_off[2], s_off[2];
#pragma unroll
    for (int sl = 0; sl < 2; ++sl) {
      const int sb = 2 * q + sl;   // slab of the 128-row item
      const uint32_t unit = ((sb >> 2) * kStageUnits + hu) * kUnitBytes;
      q_off[sl] = kPOff + unit + (sb & 3) * 512 + lane * 16;
      s_off[sl] = kPOff + unit + kUnitQBytes + (sb & 3) * 64 + g * 8;
    }
    const uint32_t t_lane = static_cast<uint32_t>(32 * q) << 16;
    int it = 0;
    for (int q = 0; !abort_flag; ++q) {
      int i = take_item(item_full, item_empty, item_q, item_f, q, a.status, nullptr);
      i = __shfl_sync(0xffffffffu, i, 0);
      if (i < 0) {
        if (i == -2) abort_flag = 1;
        break;
      }
      for (int ks = 0; ks < n_stages; ++ks, ++it) {
        if ((it % kGroups) != grp) continue;
        const int sp = it % kSP, sa = it % kSA;
        // the packed stage, and (after the first kSA stages) the A slot
        // released by the MMAs of stage it - kSA
        bool ok = it < kSA ? mbar_wait(&p_full[sp], (it / kSP) & 1, a.status)
                           : mbar_wait2(&p_full[sp], (it / kSP) & 1, &a_empty[sa], ((it / kSA) - 1) & 1, a.status);
        ok = __all_sync(0xffffffffu, ok);   // warp-uniform: the .sync.aligned work below
        if (!ok) {
          abort_flag = 1;
          break;
        }
        tc_fence_after();
        const bool active = hu < stage_units(ks, n_units);
        uint32_t v[2][16];
        if (active) dequant_two_slabs(smem + sp * kPStageBytes, q_off, s_off, mask, magic, v);
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_empty[sp]);     // packed data consumed into registers
        if (active) {
          const uint32_t col = tmem_base + kACol0 + sa * kASlotCols + hu * (kUnitK / 2);
          tmem_st_16x128b_x8(col + t_lane, v[0]);
          tmem_st_16x128b_x8(col + t_lane + (16u << 16), v[1]);
          tmem_st_wait();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&a_full[sa]);
      }
    }
  } else if (warp >= kEpiWarp0) {
    // ------------------------------------------------------------ epilogue
    const int qw = warp & 3;                 // TMEM lane quarter of this warp
    int j = 0;
    for (; !abort_flag; ++j) {
      Item item;
      int i = take_item(item_full, item_empty, item_q, item_f, j, a.status, &item);
      i = __shfl_sync(0xffffffffu, i, 0);
      if (i < 0) {
        if (i == -2) abort_flag = 1;
        break;
      }
      const int acc = j % kAccBufs, use = j / kAccBufs;
      if (!mbar_wait_backoff(&tfull_bar[acc], use & 1, a.status)) {
        abort_flag = 1;
        break;
      }
      tc_fence_after();
      const uint32_t taddr = tmem_base + acc * kAccCols + (static_cast<uint32_t>(32 * qw) << 16);
      const int row_in = 32 * qw + lane;     // A row = TMEM lane
      for (int c0 = 0; c0 < item.rows; c0 += 32) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(taddr + c0, v);
        tmem_ld_wait();
        const int ncol = min(32, item.rows - c0);
        if (a.gate_up) {
          // rows 0-7 of a 16-row slab are gate, rows 8-15 the matching up rows
          const int bt = 2 * item.wt + (row_in >> 6);
          const int p = row_in & 63;
          const int col = 32 * bt + 8 * (p >> 4) + (p & 7);
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const float mine = __uint_as_float(v[c]);
            const float other = __shfl_xor_sync(0xffffffffu, mine, 8);
            if (!(lane & 8) && c < ncol) {
              const float h = __fdividef(mine, 1.0f + __expf(-mine)) * other;
              a.C[static_cast<size_t>(item.row0 + c0 + c) * a.ldc + col] = f32_to_bf16_rn(h);
            }
          }
        } else if (a.Cf) {
          // weighted add: lane c holds row c's assignment and weight; each
          // column c of the accumulator goes, scaled, into that token's row
          const int col = kMRows * item.wt + row_in;
          int f = -1;
          float w = 0.f;
          if (lane < ncol) {
            f = ld_cg(a.sorted + item.row0 + c0 + lane);
            if (f < 0 || f >= a.M * a.topk) f = -1;
            else w = ld_cg(a.topk_w + f);
          }
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const int fc = __shfl_sync(0xffffffffu, f, c);
            const float wc = __shfl_sync(0xffffffffu, w, c);
            if (c < ncol && fc >= 0)
              atomicAdd(a.Cf + static_cast<size_t>(fc / a.topk) * a.N + col, wc * __uint_as_float(v[c]));
          }
        } else {
          const int col = kMRows * item.wt + row_in;
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            if (c < ncol)
              a.C[static_cast<size_t>(item.row0 + c0 + c) * a.ldc + col] =
                  f32_to_bf16_rn(__uint_as_float(v[c]));
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty_bar[acc]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda link).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// Activation tensor map: rows of K BF16 (row stride 2K bytes), boxes of 64
// along K by `box_rows` rows, 128-byte swizzle.
bool encode_b_map(EncodeTiledFn encode, CUtensorMap* map, const uint16_t* B, int K, size_t rows,
                  int box_rows) {
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kUnitK), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(B), dims, strides,
                box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

size_t gemm_large_smem_bytes() { return kSmemBytes; }

cudaError_t gemm_large_launch(const GemmLaunch& g, const uint16_t* B, size_t b_rows,
                              cudaStream_t st) {
  if (g.N % kMRows != 0 || g.K % kUnitK != 0 || g.E_local > kMaxExperts || b_rows < 8)
    return cudaErrorInvalidValue;
  EncodeTiledFn encode = get_encode_fn();
  if (!encode) return cudaErrorNotSupported;
  // Box heights divide 192 (the activation slot), so whole boxes never
  // overrun a slot; rows past the tensor's end read as zeros.
  int box_s = 8;
  for (int r : {64, 32, 16})
    if (b_rows >= static_cast<size_t>(r)) { box_s = r; break; }
  const int box_b = b_rows >= static_cast<size_t>(kMaxTok) ? kMaxTok : box_s;
  CUtensorMap map_s, map_b;
  if (!encode_b_map(encode, &map_s, B, g.K, b_rows, box_s) ||
      !encode_b_map(encode, &map_b, B, g.K, b_rows, box_b))
    return cudaErrorInvalidValue;
  LargeArgs a;
  a.packed = static_cast<const uint8_t*>(g.packed);
  a.counts = g.counts;
  a.offsets = g.offsets;
  a.work = g.work;
  a.C = g.C;
  a.Cf = g.epilogue == CHORD_EPI_WEIGHTED_ADD ? g.Cf : nullptr;
  a.topk_w = g.topk_w;
  a.sorted = g.sorted;
  a.M = g.M;
  a.topk = g.topk;
  a.status = g.status;
  a.N = g.N;
  a.K = g.K;
  a.E_local = g.E_local;
  const bool gate_up = g.epilogue == CHORD_EPI_SILU_MUL;
  const PackHeader h = make_pack_header(g.E_local, g.N, g.K, gate_up);
  a.n_blob_tiles = h.n_tiles;
  a.tile_bytes = h.tile_bytes;
  a.need_flags = gate_up ? kPackFlagGateUp : 0u;
  a.gate_up = gate_up ? 1 : 0;
  a.ldc = gate_up ? g.N / 2 : g.N;
  a.box_s = box_s;
  a.box_b = box_b;
  a.nib_mask = 0x000F000Fu;
  a.nib_magic = 0x43004300u;
  cudaError_t err = ensure_smem_limit<gemm_large_kernel>(kSmemBytes);
  if (err != cudaSuccess) return err;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  gemm_large_kernel<<<sms, kThreads, kSmemBytes, st>>>(map_s, map_b, a);
  return cudaGetLastError();
}

// ------------------------------------------------------------ row gather
// x_sorted[r] = x[sorted[r] / topk] for r < num_tokens_post_padded (padding
// rows become zeros), so the activation rows of an expert are contiguous for
// the tensor-map loads.
__global__ void gather_rows_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ sorted,
                                   const int32_t* __restrict__ ntpp, int topk, int sentinel, int K,
                                   uint16_t* __restrict__ out) {
  const int n = __ldg(ntpp);
  const int vec_per_row = K / 8;
  for (int r = blockIdx.x; r < n; r += gridDim.x) {
    const int f = __ldg(sorted + r);
    uint4* dst = reinterpret_cast<uint4*>(out + static_cast<size_t>(r) * K);
    if (f >= sentinel) {
      for (int c = threadIdx.x; c < vec_per_row; c += blockDim.x) dst[c] = make_uint4(0, 0, 0, 0);
    } else {
      const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<size_t>(f / topk) * K);
      for (int c = threadIdx.x; c < vec_per_row; c += blockDim.x) dst[c] = __ldg(src + c);
    }
  }
}

cudaError_t gather_rows_launch(const uint16_t* x, const int32_t* sorted, const int32_t* ntpp,
                               int topk, int sentinel, int K, size_t capacity, uint16_t* out,
                               cudaStream_t st) {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long want = static_cast<long long>(capacity);
  const int grid = static_cast<int>(want < 8LL * sms ? (want > 0 ? want : 1) : 8LL * sms);
  gather_rows_kernel<<<grid, 256, 0, st>>>(x, sorted, ntpp, topk, sentinel, K, out);
  return cudaGetLastError();
}

}  // namespace chord
