// Prefill-chunk attention on the 5th-generation tensor cores (tcgen05 + TMEM), K by TMA,
// V by 16-byte cp.async.
//
// Same causal rule as prefill.cuh ("mini_engine" README, "What it does": chunked prefill;
// "09 -- Mini Inference Engine (The Capstone)", "Week 3": mixed batches): row r of an n-row
// span sits at position ctx - n + r and sees keys 0 .. ctx - n + r.  An item is (sequence,
// tile of P = floor(128 / G) positions of its span, kv head h), and its 128-row Q tile
// stacks the G query heads that share kv head h: tile row r is position q0 + r / G of q head
// h G + r % G.  Every K/V tile is thus loaded once for the whole GQA group; rows past G P
// are idle.
//
// Per item, one CTA of sixteen warps with fixed roles:
//   warps 0, 1, 6, 7   K by TMA: warp 0 loads the Q tile once per item (3-D tensor map over
//                q); all four issue the K tiles of 128 keys gathered through the block table
//                (4-D pool map, one box per block of the tile and 64-dim half of kv head h),
//                the boxes split between them, into a 2-stage ring.  A warp issues its boxes
//                one after the other (about 140 SM clocks per box on GB300), so one warp
//                alone could not keep up with the tensor cores at 16-token blocks.
//   warps 2, 3, 5   V by 16-byte cp.async into a 3-stage ring in the 128-byte swizzled
//                layout the MMA reads; keys past the visible range are zero-filled instead
//                of loaded (0 * NaN would poison O), so no V tile needs a second pass.
//   warp 4       allocates TMEM (S: 2 x 128 columns; O: d columns; P: 2 x 64 columns) and,
//                from one thread, issues   S = Q . K^T   (M 128, N 128, K d)   and
//                                          O += P . V    (M 128, N d,   K 128)
//                as tcgen05.mma kind::f16 (S from Q and K in shared memory, O from P in TMEM
//                and V in shared memory as an MN-major operand), fp32 accumulators in TMEM,
//                completion signalled with tcgen05.commit on mbarriers.
//   warps 8-15   softmax, two threads per query row: warp w reads TMEM lanes 32 (w % 4) ..,
//                warps 8-11 the first 64 keys of each S tile, warps 12-15 the other 64.  The
//                two threads of a row exchange their partial row maxima through shared memory
//                (an mbarrier per pair of warps, bounded waits), then each computes
//                p = 2^(s scale - m) for its 64 keys, keeps its own part of the row sum l in
//                the log2 domain and writes its half of P (bf16) to TMEM, double-buffered.  O
//                in TMEM is rescaled (each thread its half of the d columns) only when the
//                row max grows by more than 2^8 (the stale max stays the reference otherwise;
//                O and l share it, so the result is unchanged).  At the end of an item the two
//                halves of l are added, O / l is read out and stored as bf16.
// Items follow one another without a CTA-wide barrier: the Q tile is reloaded once the MMA has
// read it (q_empty), and the next item's first P.V overwrites O only after the softmax warps
// have read it (o_free), so loads and products of the next item overlap the epilogue of the
// last one.  Every wait is bounded; a CTA that times out sets PKV_DEVERR_TIMEOUT and finishes
// its items without further work.
#pragma once

#include <cuda.h>

#include "decode_tc.cuh"
#include "prefill.cuh"
#include "tcgen05.cuh"

namespace pkv {

struct PrefillTcParams {
  CUtensorMap tmap_q;  // 3-D {d, Hq, T}, box {64, G, P}, 128B swizzle
  CUtensorMap tmap_k;  // 4-D {d, Hkv, block_size, num_blocks}, box {64, 1, block_size, 1}, 128B swizzle
  PrefillParams p;
  int group;  // G = Hq / Hkv
  int prows;  // P = floor(128 / G): positions per item
};

template <int D>
struct PrefillTcCfg {
  static constexpr int kThreads = 512;
  static constexpr int BQ = 128;  // query rows per item
  static constexpr int BK = 128;  // keys per K/V tile
  static constexpr int HALVES = D / 64;
  static constexpr int CH = D / 8;        // 16-byte chunks per K/V row
  static constexpr int kBlk = 128 * 128;  // one [128 rows][64 elements] swizzled block: 16 KB
  static constexpr int kQBytes = BQ * D * 2;
  static constexpr int kKVBytes = BK * D * 2;
  static constexpr int KST = 2;  // K ring stages
  static constexpr int VST = 3;  // V ring stages
  static constexpr int kKWarps = 4;      // K box issuers (warps 0, 1, 6, 7)
  static constexpr int kVThreads = 96;   // V loader threads (warps 2, 3, 5)
  static constexpr int kVRounds = (BK * CH + kVThreads - 1) / kVThreads;  // 16-byte chunks per V loader per tile (at most)
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + kQBytes;
  static constexpr int OFF_V = OFF_K + KST * kKVBytes;
  static constexpr int OFF_X = OFF_V + VST * kKVBytes;  // row-max exchange: [2][4][2][32] floats
  static constexpr int OFF_BAR = OFF_X + 2 * 4 * 2 * 32 * 4;
  static constexpr int kSmemBytes = OFF_BAR + 512 + 1024;  // + barriers + alignment slack
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t COL_O = 256;  // O: D columns
  static constexpr uint32_t COL_P = 384;  // P (bf16 pairs): 2 buffers x 64 columns
  static_assert(D <= 128, "TMEM columns: S 2 x 128, O D, P 2 x 64");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
  static_assert(kVThreads % CH == 0, "each V loader copies one chunk column");
};

__device__ __forceinline__ void tma_load_3d(void* dst_smem, const CUtensorMap* map, int c0, int c1, int c2,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst_smem)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

// 16-byte global -> shared copy that fills the destination with zeros when `valid` is false
// (src_size 0: nothing is read from `src`, which must still be a valid address).
__device__ __forceinline__ void cp_async_16_zfill(uint32_t dst_smem, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst_smem), "l"(src), "r"(valid ? 16 : 0)
               : "memory");
}

// Two fp32 lanes per instruction (packed f32x2 FMA and add, Blackwell).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 r;
  asm("{\n\t.reg .b64 a, b, c, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\tmov.b64 c, {%6, %7};\n\t"
      "fma.rn.f32x2 d, a, b, c;\n\tmov.b64 {%0, %1}, d;\n\t}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return r;
}
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
  float2 r;
  asm("{\n\t.reg .b64 a, b, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
      "add.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;\n\t}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}

// All 32 lanes wait; the outcome is made warp-uniform (any lane timing out aborts the warp).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, unsigned int* err,
                                          volatile int* abort_flag) {
  const bool ok = wait_or_abort(bar, parity, err, abort_flag);
  return __all_sync(0xffffffffu, ok);
}

// The work item a CTA takes in a wave, and what every role needs to know about it.
struct PfItem {
  int h;        // kv head; q heads h G .. h G + G - 1
  int b;        // sequence
  int s0;       // first query row of the span
  int q0;       // first position of the item within the span
  int qrows;    // positions of this item
  int pos0;     // position of the item's first row
  int kv_end;   // keys [0, kv_end) are visible to some row
  int nkt;      // K/V tiles of 128 keys
};

__device__ __forceinline__ PfItem pf_item(const PrefillParams& p, int item, int PR) {
  PfItem it;
  const int ti = item / p.hkv;
  it.h = item - ti * p.hkv;
  it.b = p.plan.pf_seq[ti];
  const int j = p.plan.pf_tile[ti];
  it.s0 = p.qsl[it.b];
  const int n = p.qsl[it.b + 1] - it.s0;
  const int ctx = p.context_lens[it.b];
  it.q0 = j * PR;
  it.qrows = min(PR, n - it.q0);
  it.pos0 = ctx - n + it.q0;
  it.kv_end = it.pos0 + it.qrows;
  it.nkt = ceil_div(it.kv_end, 128);
  return it;
}

template <int D>
__global__ void __launch_bounds__(512, 1) prefill_tc_kernel(const __grid_constant__ PrefillTcParams P) {
  using C = PrefillTcCfg<D>;
  constexpr int HALVES = C::HALVES;
  const PrefillParams& p = P.p;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  float* xch = reinterpret_cast<float*>(smem + C::OFF_X);  // [parity][quarter][half][lane]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars + 0;
  uint64_t* q_empty = bars + 1;   // the MMA finished reading the Q tile
  uint64_t* k_full = bars + 2;    // [KST]
  uint64_t* k_empty = bars + 4;   // [KST] the QK MMA finished reading the K stage
  uint64_t* v_full = bars + 6;    // [VST]
  uint64_t* v_empty = bars + 9;   // [VST] the P.V MMA finished reading the V stage
  uint64_t* s_full = bars + 12;   // [2] S buffer written
  uint64_t* s_free = bars + 14;   // [2] softmax finished reading the S buffer
  uint64_t* p_full = bars + 16;   // [2] P buffer written
  uint64_t* pv_done = bars + 18;  // [2] P.V of the tile whose P is in that buffer completed
  uint64_t* o_free = bars + 20;   // the softmax finished reading an item's O
  uint64_t* xbar = bars + 21;     // [4] row-max exchange of the two softmax warps of a quarter
  uint64_t* fin = bars + 25;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 26);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 27);
  static_assert(C::KST == 2 && C::VST == 3, "barrier layout");
  // P.V of tile t completes pv_done[t % 2] for the (t / 2)-th time
  auto pv_wait = [&](int t) { return warp_wait(&pv_done[t & 1], (t >> 1) & 1, p.err, abort_flag); };
  const float NEG_INF = -__int_as_float(0x7f800000);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int s = 0; s < C::KST; ++s) {
      mbar_init(&k_full[s], C::kKWarps);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < C::VST; ++s) {
      mbar_init(&v_full[s], C::kVThreads);
      mbar_init(&v_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&s_free[s], 8);
      mbar_init(&p_full[s], 8);
      mbar_init(&pv_done[s], 1);
    }
    mbar_init(o_free, 8);
    for (int s = 0; s < 4; ++s) mbar_init(&xbar[s], 64);
    mbar_init(fin, 1);
    fence_mbar_init();
    *abort_flag = 0;
  }
  if (warp == 0 && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&P.tmap_q)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&P.tmap_k)) : "memory");
  }
  // TMEM is taken while the planner still runs (this kernel starts early under programmatic
  // dependent launch), so the allocation is off the critical path.
  if (warp == 4) {
    tc5::alloc(tmem_slot, C::TMEM_COLS);
    tc5::relinquish();
  }
  tc5::fence_before();
  __syncthreads();
  tc5::fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();  // the tile list is written by the planner kernel (on a second stream an event orders it)
  pdl_trigger();
  const int n_tiles = p.plan.header[3];
  const int total = n_tiles * p.hkv;
  // CTAs that take items: the planner's count, fewer than launched when the prefill shares
  // the SMs with the decode.  A CTA past it, or whose first snake-order slot is past the
  // item list (every later slot is at least nact), has no item in any wave: it gives TMEM
  // back and leaves.  On a batch without prefill spans that is every CTA.
  const int nact = min(max(p.plan.header[5], 0), static_cast<int>(gridDim.x));
  if (static_cast<int>(blockIdx.x) >= total || static_cast<int>(blockIdx.x) >= nact) {
    if (warp == 4) tc5::dealloc(tmem, C::TMEM_COLS);
    return;
  }
  const int G = P.group;
  const int PR = P.prows;
  const int bs_log2 = p.bs_log2;
  const int bs = 1 << bs_log2;

  if (warp < 2 || warp == 6 || warp == 7) {
    // ------------------------------------- Q (warp 0) and K tiles by TMA (warps 0, 1, 6, 7)
    // A tile's boxes are numbered lbox * HALVES + half (lbox: block within the tile); box x
    // goes to K warp x % 4, lane x / 4.  The block id of a lane's box is read two tiles before
    // its load, so the table reads never sit between a freed stage and its refill.
    const uint64_t pol = l2_policy_evict_last();  // K tiles are re-read by the other items
    const int kw = warp < 2 ? warp : warp - 4;
    const int bx = C::kKWarps * lane + kw;
    const int lbox = bx / HALVES, lhalf = bx - lbox * HALVES;
    const bool lane_boxes = lbox < C::BK / bs;
    bool ok = !*abort_flag;
    int t_glob = 0, item_no = 0;
    for (int wave = 0; wave * nact < total && ok; ++wave) {
      const int ord = snake_order(wave, blockIdx.x, nact);
      if (ord >= total) continue;
      const PfItem it = pf_item(p, total - 1 - ord, PR);
      if (warp == 0) {
        if (item_no > 0) ok = warp_wait(q_empty, (item_no - 1) & 1, p.err, abort_flag);
        if (!ok) break;
        if (lane == 0) mbar_arrive_expect_tx(q_full, static_cast<uint32_t>(HALVES * G * PR * 128));
        __syncwarp();
        if (lane < HALVES)
          tma_load_3d(smem + C::OFF_Q + lane * C::kBlk, &P.tmap_q, lane * 64, it.h * G, it.s0 + it.q0, q_full);
      }
      const int32_t* btrow = p.block_tables + static_cast<int64_t>(it.b) * p.bt_stride;
      auto fetch_block = [&](int jt) -> int {
        const int key0 = jt * C::BK + lbox * bs;
        return (jt < it.nkt && lane_boxes && key0 < it.kv_end) ? btrow[key0 >> bs_log2] : 0;
      };
      int nb0 = fetch_block(0), nb1 = fetch_block(1);
      for (int jt = 0; jt < it.nkt; ++jt) {
        const int f = t_glob + jt;
        const int ks = f % C::KST;
        int blk = nb0;
        nb0 = nb1;
        nb1 = fetch_block(jt + 2);
        if (f >= C::KST) {
          ok = warp_wait(&k_empty[ks], (f / C::KST - 1) & 1, p.err, abort_flag);
          if (!ok) break;
        }
        // boxes past kv_end are not loaded (their block may not exist, and those keys are
        // never used); each warp expects the bytes of its own boxes
        const int nbox = ceil_div(min(C::BK, it.kv_end - jt * C::BK), bs);
        const bool mine = lane_boxes && lbox < nbox;
        const unsigned nmine = __popc(__ballot_sync(0xffffffffu, mine));
        if (lane == 0) mbar_arrive_expect_tx(&k_full[ks], nmine * static_cast<uint32_t>(bs * 128));
        __syncwarp();
        if (mine) {
          if (blk < 0 || blk >= p.num_blocks) {
            raise_error(p.err, PKV_DEVERR_BLOCK_RANGE);
            blk = 0;
          }
          unsigned char* dst = smem + C::OFF_K + ks * C::kKVBytes + lhalf * C::kBlk + lbox * bs * 128;
          tma_load_4d(dst, &P.tmap_k, lhalf * 64, it.h, 0, blk, &k_full[ks], pol);
        }
      }
      t_glob += it.nkt;
      ++item_no;
    }
  }
  else if (warp == 4) {
    // ---------------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdescQK = tc5::idesc_bf16_f32(128, 128);
      constexpr uint32_t kIdescPV = tc5::idesc_bf16_f32(128, D, true);
      bool ok = !*abort_flag;
      int t_glob = 0, item_no = 0;
      // O += P . V of tile fp; the first of an item overwrites O, once the softmax warps have
      // read the previous item's O
      auto issue_pv = [&](int fp, bool first) -> bool {
        if (!wait_or_abort(&v_full[fp % C::VST], (fp / C::VST) & 1, p.err, abort_flag)) return false;
        if (!wait_or_abort(&p_full[fp & 1], (fp >> 1) & 1, p.err, abort_flag)) return false;
        if (first && item_no > 0 && !wait_or_abort(o_free, (item_no - 1) & 1, p.err, abort_flag)) return false;
        tc5::fence_after();
        const uint32_t vst = sb + C::OFF_V + (fp % C::VST) * C::kKVBytes;
#pragma unroll
        for (int kk = 0; kk < C::BK / 16; ++kk)  // A = P from TMEM: 16 keys = 8 columns
          tc5::mma_ts(tmem + C::COL_O, tmem + C::COL_P + 64u * (fp & 1) + 8u * kk,
                      tc5::smem_desc_mn128(vst + kk * 2048, C::kBlk), kIdescPV, (first && kk == 0) ? 0u : 1u);
        tc5::commit(&pv_done[fp & 1]);
        tc5::commit(&v_empty[fp % C::VST]);
        return true;
      };
      for (int wave = 0; wave * nact < total && ok; ++wave) {
        const int ord = snake_order(wave, blockIdx.x, nact);
        if (ord >= total) continue;
        const PfItem it = pf_item(p, total - 1 - ord, PR);
        ok = wait_or_abort(q_full, item_no & 1, p.err, abort_flag);
        for (int jt = 0; jt < it.nkt && ok; ++jt) {
          const int f = t_glob + jt;
          const int s = f & 1;  // S buffer
          const int ks = f % C::KST;
          ok = wait_or_abort(&k_full[ks], (f / C::KST) & 1, p.err, abort_flag);
          if (ok && f >= 2) ok = wait_or_abort(&s_free[s], ((f >> 1) - 1) & 1, p.err, abort_flag);
          if (!ok) break;
          tc5::fence_after();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * C::kBlk + (kk & 3) * 32;
            tc5::mma_ss(tmem + 128u * s, tc5::smem_desc_k128(sb + C::OFF_Q + off),
                        tc5::smem_desc_k128(sb + C::OFF_K + ks * C::kKVBytes + off), kIdescQK, kk > 0 ? 1u : 0u);
          }
          tc5::commit(&s_full[s]);
          tc5::commit(&k_empty[ks]);
          if (jt == it.nkt - 1) tc5::commit(q_empty);  // the item's last read of Q
          if (jt > 0) ok = issue_pv(f - 1, jt == 1);
        }
        if (ok) ok = issue_pv(t_glob + it.nkt - 1, it.nkt == 1);
        t_glob += it.nkt;
        ++item_no;
      }
    }
    __syncwarp();
  }
  else if (warp == 2 || warp == 3 || warp == 5) {
    // ------------------------------------------------------- V tiles by cp.async (3 warps)
    // Thread v (0..95) copies chunks c = v + 96 i of a tile: row c / CH, 16-byte chunk
    // c % CH of that row (its 64-dim half and the chunk within it), to the position the
    // 128-byte swizzle gives it.  The tile's block ids (128 / block_size of them) are read by
    // the first lanes of each loader warp two tiles ahead and handed out by shuffles.  Each
    // thread keeps two tiles in flight: after committing tile f it waits for tile f - 1,
    // fences it for the tensor cores (async proxy) and arrives on that stage's full barrier.
    const int vt = warp < 4 ? warp - 2 : 2;
    const int tv = vt * 32 + lane;
    const int ch = tv % C::CH;  // the same chunk column in every row this thread copies
    const int half = ch >> 3, c8 = ch & 7;
    const int nblk = C::BK >> bs_log2;  // blocks per tile (1 .. 16)
    bool ok = !*abort_flag;
    int t_glob = 0, pending = -1;
    for (int wave = 0; wave * nact < total && ok; ++wave) {
      const int ord = snake_order(wave, blockIdx.x, nact);
      if (ord >= total) continue;
      const PfItem it = pf_item(p, total - 1 - ord, PR);
      const int32_t* btrow = p.block_tables + static_cast<int64_t>(it.b) * p.bt_stride;
      auto fetch_ids = [&](int jt) -> int {
        const int key0 = jt * C::BK + lane * bs;
        int blk = (jt < it.nkt && lane < nblk && key0 < it.kv_end) ? btrow[key0 >> bs_log2] : 0;
        return blk;
      };
      int id0 = fetch_ids(0), id1 = fetch_ids(1);
      const bf16* vh = p.v_cache + static_cast<int64_t>(it.h) * D + ch * 8;
      for (int jt = 0; jt < it.nkt; ++jt) {
        const int f = t_glob + jt;
        const int vs = f % C::VST;
        int ids = id0;
        id0 = id1;
        id1 = fetch_ids(jt + 2);
        if (f >= C::VST) {
          ok = warp_wait(&v_empty[vs], (f / C::VST - 1) & 1, p.err, abort_flag);
          if (!ok) break;
        }
        if (ids < 0 || ids >= p.num_blocks) {
          if (vt == 0) raise_error(p.err, PKV_DEVERR_BLOCK_RANGE);
          ids = 0;
        }
        const uint32_t vbase = sb + C::OFF_V + vs * C::kKVBytes + half * C::kBlk;
#pragma unroll
        for (int i = 0; i < C::kVRounds; ++i) {
          if (tv + C::kVThreads * i >= C::BK * C::CH) break;
          const int row = (tv + C::kVThreads * i) / C::CH;
          const int key = jt * C::BK + row;
          const bool valid = key < it.kv_end;
          const int blk = __shfl_sync(0xffffffffu, ids, row >> bs_log2);
          const bf16* src =
              valid ? vh + ((static_cast<int64_t>(blk) << bs_log2) + (key & (bs - 1))) * p.hkv * D : p.v_cache;
          cp_async_16_zfill(vbase + row * 128 + ((c8 ^ (row & 7)) << 4), src, valid);
        }
        cp_async_commit();
        if (pending >= 0) {
          cp_async_wait<1>();
          fence_proxy_async_smem();
          mbar_arrive(&v_full[pending % C::VST]);
        }
        pending = f;
      }
      t_glob += it.nkt;
    }
    cp_async_wait<0>();  // nothing may still be landing in shared memory when the CTA leaves
    if (ok && pending >= 0) {
      fence_proxy_async_smem();
      mbar_arrive(&v_full[pending % C::VST]);
    }
  }
  else if (warp >= 8) {
    // ------------------------------------------------------------ softmax (two threads a row)
    const int qq = warp & 3;             // TMEM lanes 32 qq .. 32 qq + 31
    const int half = (warp - 8) >> 2;    // keys 64 half .. 64 half + 63 of each S tile
    const int r = 32 * qq + lane;        // query row of the tile
    const int rt = r / G;                // position within the item
    const int rg = r - rt * G;           // q head within the group
    const uint32_t trow = tmem + (static_cast<uint32_t>(32 * qq) << 16);
    float* my_x = xch + (qq * 2 + half) * 32 + lane;        // + parity * 256
    const float* other_x = xch + (qq * 2 + (1 - half)) * 32 + lane;
    int xph = 0;  // exchanges done by this pair of warps
    // both threads of a row publish a value and read the other's (bounded wait on the pair's
    // barrier; two slots by parity, so a thread one exchange ahead never overwrites a value
    // its partner has yet to read)
    auto exchange = [&](float mine, float& other) -> bool {
      my_x[(xph & 1) * 256] = mine;
      mbar_arrive(&xbar[qq]);
      const bool okx = warp_wait(&xbar[qq], xph & 1, p.err, abort_flag);
      other = other_x[(xph & 1) * 256];
      ++xph;
      return okx;
    };
    bool ok = !*abort_flag;
    int t_glob = 0;
    for (int wave = 0; wave * nact < total && ok; ++wave) {
      const int ord = snake_order(wave, blockIdx.x, nact);
      if (ord >= total) continue;
      const PfItem it = pf_item(p, total - 1 - ord, PR);
      const bool live = rt < it.qrows;  // (rt < qrows implies r < G P)
      const int pos = it.pos0 + rt;
      float m_run = NEG_INF, l_run = 0.f;  // l_run: this thread's half of the row sum
      for (int jt = 0; jt < it.nkt && ok; ++jt) {
        const int f = t_glob + jt;
        const int s = f & 1;
        ok = warp_wait(&s_full[s], (f >> 1) & 1, p.err, abort_flag);
        if (!ok) break;
        tc5::fence_after();
        float sc[64];
        tc5::ld32(trow + 128u * s + 64u * half, *reinterpret_cast<float(*)[32]>(sc));
        tc5::ld32(trow + 128u * s + 64u * half + 32u, *reinterpret_cast<float(*)[32]>(sc + 32));
        tc5::wait_ld();
        tc5::fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_free[s]);
        // row max of the raw scores over eight partial maxima (qscale > 0 keeps the order); the
        // mask is a select and only the diagonal tiles need it
        const int key0 = jt * C::BK + 64 * half;
        float mx8[8];
#pragma unroll
        for (int x = 0; x < 8; ++x) mx8[x] = NEG_INF;
        if (live && key0 + 63 <= pos) {
#pragma unroll
          for (int c = 0; c < 64; ++c) mx8[c & 7] = fmaxf(mx8[c & 7], sc[c]);
        } else {
#pragma unroll
          for (int c = 0; c < 64; ++c) {
            sc[c] = (live && key0 + c <= pos) ? sc[c] : NEG_INF;
            mx8[c & 7] = fmaxf(mx8[c & 7], sc[c]);
          }
        }
        const float mine = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                 fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
        float other;
        ok = exchange(mine, other);
        if (!ok) break;
        // the same operands in the same order in both threads: the same max, bit for bit
        const float mraw = half == 0 ? fmaxf(mine, other) : fmaxf(other, mine);
        const float mx = mraw * p.qscale;  // -inf stays -inf
        float corr = 1.f;
        bool resc = false;
        if (m_run == NEG_INF) {
          m_run = mx;  // nothing accumulated for this row yet
        } else if (mx > m_run + 8.f) {
          corr = fast_exp2(m_run - mx);
          m_run = mx;
          resc = true;
        }
        const float base = m_run == NEG_INF ? 0.f : m_run;
        // p = 2^(s * qscale - base): one ex2 per score, the FMA and the partial sums on packed
        // f32x2 pairs
        const float2 qs2 = make_float2(p.qscale, p.qscale);
        const float2 nb2 = make_float2(-base, -base);
        float2 ls4[4];
#pragma unroll
        for (int x = 0; x < 4; ++x) ls4[x] = make_float2(0.f, 0.f);
#pragma unroll
        for (int c = 0; c < 64; c += 2) {
          const float2 t = ffma2(make_float2(sc[c], sc[c + 1]), qs2, nb2);
          sc[c] = fast_exp2(t.x);
          sc[c + 1] = fast_exp2(t.y);
          ls4[(c >> 1) & 3] = fadd2(ls4[(c >> 1) & 3], make_float2(sc[c], sc[c + 1]));
        }
        const float2 ls2 = fadd2(fadd2(ls4[0], ls4[1]), fadd2(ls4[2], ls4[3]));
        l_run = l_run * corr + (ls2.x + ls2.y);
        if (jt > 0 && __any_sync(0xffffffffu, resc)) {
          // this thread's half of the row of O is rescaled once every P.V issued so far has
          // landed in it
          ok = pv_wait(f - 1);
          if (!ok) break;
          tc5::fence_after();
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {  // 16 columns at a time: the 64 scores stay live
            float o[16];
            const uint32_t col = C::COL_O + (D / 2) * half + 16u * c;
            tc5::ld16(trow + col, o);
            tc5::wait_ld();
#pragma unroll
            for (int x = 0; x < 16; ++x) o[x] *= corr;
            tc5::st16(trow + col, o);
          }
          tc5::wait_st();
        }
        if (f >= 2) {  // this P buffer was read by the P.V of tile f - 2
          ok = pv_wait(f - 2);
          if (!ok) break;
          tc5::fence_after();
        }
        // this half of the P row as bf16 pairs into TMEM, the A operand of P.V: column c of
        // the buffer holds keys 2c, 2c + 1
        // (packed in place: pair x goes to sc[x] once sc[2x] and sc[2x + 1] are read)
#pragma unroll
        for (int x = 0; x < 32; ++x) sc[x] = __uint_as_float(pack_bf16x2(sc[2 * x], sc[2 * x + 1]));
        tc5::st32(trow + C::COL_P + 64u * (f & 1) + 32u * half, *reinterpret_cast<const float(*)[32]>(sc));
        tc5::wait_st();
        tc5::fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[f & 1]);
      }
      // epilogue: the full row sum, then this thread's half of O / l as bf16
      if (ok) ok = pv_wait(t_glob + it.nkt - 1);
      float l_other = 0.f;
      if (ok) ok = exchange(l_run, l_other);
      if (ok) {
        const float l = half == 0 ? l_run + l_other : l_other + l_run;
        tc5::fence_after();
        const float inv = live ? 1.f / l : 0.f;
        bf16* orow = p.out + static_cast<int64_t>(it.s0 + it.q0 + rt) * p.o_st +
                     static_cast<int64_t>(it.h * G + rg) * p.o_sh + (D / 2) * half;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          float o[16];
          tc5::ld16(trow + C::COL_O + (D / 2) * half + 16u * c, o);
          tc5::wait_ld();
          if (live) {
#pragma unroll
            for (int x = 0; x < 2; ++x) {
              uint4 u;
              u.x = pack_bf16x2(o[8 * x + 0] * inv, o[8 * x + 1] * inv);
              u.y = pack_bf16x2(o[8 * x + 2] * inv, o[8 * x + 3] * inv);
              u.z = pack_bf16x2(o[8 * x + 4] * inv, o[8 * x + 5] * inv);
              u.w = pack_bf16x2(o[8 * x + 6] * inv, o[8 * x + 7] * inv);
              *reinterpret_cast<uint4*>(orow + 16 * c + 8 * x) = u;
            }
          }
        }
        tc5::fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(o_free);  // the next item's first P.V may overwrite O
      }
      t_glob += it.nkt;
    }
  }

  // teardown: every role is done; no MMA may still be in flight when TMEM is released
  __syncthreads();
  if (warp == 4) {
    if (lane == 0) {
      tc5::commit(fin);
      mbar_wait(fin, 0, p.err);  // bounded, and not skipped after an abort
    }
    __syncwarp();
    tc5::fence_after();
    tc5::dealloc(tmem, C::TMEM_COLS);
  }
}

}  // namespace pkv
