// Prefill-chunk attention on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// Same causal rule as prefill.cuh ("mini_engine" README, "What it does": chunked prefill;
// "09 -- Mini Inference Engine (The Capstone)", "Week 3": mixed batches): row r of an n-row
// span sits at position ctx - n + r and sees keys 0 .. ctx - n + r.  An item is (sequence,
// tile of P = floor(128 / G) positions of its span, kv head h), and its 128-row Q tile
// stacks the G query heads that share kv head h: tile row r is position q0 + r / G of q head
// h G + r % G.  Every K/V tile is thus loaded once for the whole GQA group (G = 2: half the
// K/V traffic of one item per q head); rows past G P are idle.
//
// Per item, one CTA of eight warps with fixed roles:
//   warp 0     TMA producer: the Q tile once (3-D tensor map over q), then the K tiles of
//              128 keys gathered through the block table (4-D pool map, one box per block
//              of the tile x 64 dims of kv head h), into a 3-stage ring.
//   warp 1     allocates TMEM (S: 2 x 128 columns; O: d columns; P: 2 x 64 columns) and, from one
//              thread, issues   S = Q . K^T   (M 128, N 128, K d)   and
//                               O += P . V    (M 128, N d,   K 128)  as tcgen05.mma kind::f16,
//              S from Q and K in shared memory (K-major), O from P in TMEM and V in shared
//              memory (read as it lands, an MN-major operand), fp32 accumulators in TMEM,
//              completion signalled with tcgen05.commit on mbarriers.
//   warp 3     loads the V tiles the same way into their own 3-stage ring, so neither ring
//              waits for the other.
//   warp 2     releases each V tile to the MMA, in an item's last tile after zeroing the rows
//              of keys past the visible range (unloaded or past the context: 0 * NaN would
//              poison O).
//   warps 4-7  softmax: thread = query row.  Reads its S row from TMEM, masks by select,
//              keeps a running max m and sum l in the log2 domain and writes P (bf16) back to
//              TMEM, double-buffered, so P of tile f + 1 never waits for P.V of tile f.  O in TMEM is rescaled only when the row max grows by more
//              than 2^8 (the stale max stays the reference otherwise; O and l share it, so the
//              result is unchanged).  At the end it reads O, divides by l and stores bf16.
// A CTA's items follow one another without a CTA barrier: the K and V rings, the S and P
// buffers and their barrier phases run on across items, the next item's Q tile is loaded once
// every QK of the current one has completed (q_empty), and its first P.V, which overwrites O,
// waits until the current item's epilogue has read O (o_free); so the next item's loads, QK and
// first softmax overlap the current item's last tiles and epilogue.
// Every wait is bounded; a CTA that times out sets PKV_DEVERR_TIMEOUT and finishes its items
// without further work.
#pragma once

#include <cuda.h>

#include "decode_tc.cuh"
#include "prefill.cuh"
#include "tcgen05.cuh"

namespace pkv {

struct PrefillTcParams {
  CUtensorMap tmap_q;  // 3-D {d, Hq, T}, box {64, G, P}, 128B swizzle
  CUtensorMap tmap_k;  // 4-D {d, Hkv, block_size, num_blocks}, box {64, 1, block_size, 1}, 128B swizzle
  CUtensorMap tmap_v;
  PrefillParams p;
  int group;  // G = Hq / Hkv
  int prows;  // P = floor(128 / G): positions per item
};

template <int D>
struct PrefillTcCfg {
  static constexpr int BQ = 128;  // query rows per item
  static constexpr int BK = 128;  // keys per K/V tile (8 pages)
  static constexpr int HALVES = D / 64;
  static constexpr int kBlk = 128 * 128;  // one [128 rows][64 elements] swizzled block: 16 KB
  static constexpr int kQBytes = BQ * D * 2;
  static constexpr int kKVBytes = BK * D * 2;
  static constexpr int OFF_Q = 0;
  static constexpr int KST = 3;  // K ring stages: a K tile is requested two tiles ahead of its QK
  static constexpr int VST = 3;  // V ring stages
  static constexpr int OFF_K = OFF_Q + kQBytes;
  static constexpr int OFF_V = OFF_K + KST * kKVBytes;
  static constexpr int OFF_BAR = OFF_V + VST * kKVBytes;
  static constexpr int kSmemBytes = OFF_BAR + 256 + 1024;  // + barriers + alignment slack
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t COL_O = 256;  // O: D columns
  static constexpr uint32_t COL_P = 384;  // P (bf16 pairs): 2 buffers x 64 columns
  static_assert(D <= 128, "TMEM columns: S 2 x 128, O D, P 2 x 64");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

__device__ __forceinline__ void tma_load_3d(void* dst_smem, const CUtensorMap* map, int c0, int c1, int c2,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst_smem)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
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

template <int D>
__global__ void __launch_bounds__(256, 1) prefill_tc_kernel(const __grid_constant__ PrefillTcParams P) {
  using C = PrefillTcCfg<D>;
  constexpr int HALVES = C::HALVES;
  const PrefillParams& p = P.p;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars + 0;
  uint64_t* k_full = bars + 1;    // [KST]
  uint64_t* k_empty = bars + 4;   // [KST] MMA finished reading the K stage
  uint64_t* v_full = bars + 7;    // [VST]
  uint64_t* v_empty = bars + 10;  // [VST] the P.V MMA finished reading the V stage
  uint64_t* s_full = bars + 13;   // [2] S buffer written
  uint64_t* s_free = bars + 15;   // [2] softmax finished reading the S buffer
  uint64_t* vt_full = bars + 17;  // V tile released to the MMA
  uint64_t* p_full = bars + 18;   // [2] P buffer written
  uint64_t* pv_done = bars + 20;  // [2] P.V of the tile whose P is in that buffer completed
  uint64_t* fin = bars + 22;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 23);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 24);
  uint64_t* q_empty = bars + 25;  // every QK of an item completed: its Q tile may be replaced
  uint64_t* o_free = bars + 26;   // the item's epilogue read O: the next item's P.V may write it
  static_assert(C::KST == 3 && C::VST == 3, "barrier layout");
  // P.V of tile t completes pv_done[t % 2] for the (t / 2)-th time
  auto pv_wait = [&](int t) { return warp_wait(&pv_done[t & 1], (t >> 1) & 1, p.err, abort_flag); };
  const float NEG_INF = -__int_as_float(0x7f800000);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < C::KST; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < C::VST; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&s_free[s], 4);
    }
    mbar_init(vt_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&p_full[s], 4);
      mbar_init(&pv_done[s], 1);
    }
    mbar_init(fin, 1);
    mbar_init(q_empty, 1);
    mbar_init(o_free, 4);
    fence_mbar_init();
    *abort_flag = 0;
  }
  if (warp == 0 && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&P.tmap_q)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&P.tmap_k)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&P.tmap_v)) : "memory");
  }
  // TMEM is taken while the planner still runs (this kernel starts early under programmatic
  // dependent launch), so the allocation is off the critical path.
  if (warp == 1) {
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
    if (warp == 1) tc5::dealloc(tmem, C::TMEM_COLS);
    return;
  }
  const int G = P.group;
  const int PR = P.prows;
  const uint64_t pol = l2_policy_evict_last();  // K/V tiles are re-read by the other items

  int t_glob = 0;  // K/V tiles this CTA has processed (ring slots, S buffers, PV phases)
  int item_no = 0;
  for (int wave = 0; wave * nact < total; ++wave) {
    const int ord = snake_order(wave, blockIdx.x, nact);
    if (ord >= total) continue;
    const int item = total - 1 - ord;  // later (longer) tiles of each span first
    const int ti = item / p.hkv;
    const int h = item - ti * p.hkv;  // kv head; q heads h G .. h G + G - 1
    const int b = p.plan.pf_seq[ti];
    const int j = p.plan.pf_tile[ti];
    const int s0 = p.qsl[b];
    const int n = p.qsl[b + 1] - s0;
    const int ctx = p.context_lens[b];
    const int q0 = j * PR;
    const int qrows = min(PR, n - q0);  // positions of this item
    const int pos0 = ctx - n + q0;
    const int kv_end = pos0 + qrows;  // keys [0, kv_end) are visible to some row
    const int nkt = ceil_div(kv_end, C::BK);

    // One K or V tile of 128 keys, issued by one warp: 128 / bs boxes of one whole block
    // (bs = block_size rows; 128 is a multiple of every block size) of kv head h per 64-dim
    // half, lane = box x half.  A box past kv_end is not loaded (its block may not exist, and
    // those keys are never used).  Larger blocks mean fewer, taller boxes.  The block id of a
    // lane's box is read by fetch_block two tiles before load_tile uses it, so the table reads
    // never sit between a freed stage and its refill.
    const int bs = 1 << p.bs_log2;
    const int lbox = lane / HALVES;  // this lane's box within a tile
    const int lhalf = lane - lbox * HALVES;
    const bool lane_loads = lbox < C::BK / bs;
    const int32_t* btrow = p.block_tables + static_cast<int64_t>(b) * p.bt_stride;
    auto fetch_block = [&](int jt) -> int {
      const int key0 = jt * C::BK + lbox * bs;
      return (jt < nkt && lane_loads && key0 < kv_end) ? btrow[key0 >> p.bs_log2] : 0;
    };
    auto load_tile = [&](bool is_v, int jt, int s, int blk) {
      const int nbox = ceil_div(min(C::BK, kv_end - jt * C::BK), bs);
      uint64_t* bar = is_v ? &v_full[s] : &k_full[s];
      if (lane == 0) mbar_arrive_expect_tx(bar, static_cast<uint32_t>(nbox * bs * 128 * HALVES));
      __syncwarp();
      if (lane_loads && lbox < nbox) {
        if (blk < 0 || blk >= p.num_blocks) {
          raise_error(p.err, PKV_DEVERR_BLOCK_RANGE);
          blk = 0;
        }
        unsigned char* dst = smem + (is_v ? C::OFF_V : C::OFF_K) + s * C::kKVBytes + lhalf * C::kBlk + lbox * bs * 128;
        tma_load_4d(dst, is_v ? &P.tmap_v : &P.tmap_k, lhalf * 64, h, 0, blk, bar, pol);
      }
    };

    if (warp == 0) {
      // ---------------------------------------------------------- TMA producer: Q and K
      // (items follow one another without a CTA barrier: the next item's Q replaces this one
      // once every QK of this item has completed, and its K tiles follow in the same ring)
      bool ok = !*abort_flag;
      if (ok && item_no > 0) ok = warp_wait(q_empty, (item_no - 1) & 1, p.err, abort_flag);
      if (ok) {
        if (lane == 0) mbar_arrive_expect_tx(q_full, static_cast<uint32_t>(HALVES * G * PR * 128));
        __syncwarp();
        if (lane < HALVES)
          tma_load_3d(smem + C::OFF_Q + lane * C::kBlk, &P.tmap_q, lane * 64, h * G, s0 + q0, q_full);
      }
      int nb0 = fetch_block(0), nb1 = fetch_block(1);
      for (int jt = 0; jt < nkt && ok; ++jt) {
        const int f = t_glob + jt;
        const int ks = f % C::KST;
        const int cur = nb0;
        nb0 = nb1;
        nb1 = fetch_block(jt + 2);
        if (f >= C::KST) {
          ok = warp_wait(&k_empty[ks], (f / C::KST - 1) & 1, p.err, abort_flag);
          if (!ok) break;
        }
        load_tile(false, jt, ks, cur);
      }
    } else if (warp == 1) {
      // ------------------------------------------------------------------- MMA issuer
      if (lane == 0) {
        constexpr uint32_t kIdescQK = tc5::idesc_bf16_f32(128, 128);
        constexpr uint32_t kIdescPV = tc5::idesc_bf16_f32(128, D, true);
        bool ok = wait_or_abort(q_full, item_no & 1, p.err, abort_flag);
        auto issue_pv = [&](int fp, bool first) -> bool {
          if (!wait_or_abort(vt_full, fp & 1, p.err, abort_flag)) return false;
          if (!wait_or_abort(&p_full[fp & 1], (fp >> 1) & 1, p.err, abort_flag)) return false;
          // the item's first P.V overwrites O: the previous item's epilogue must have read it
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
        for (int jt = 0; jt < nkt && ok; ++jt) {
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
          if (jt == nkt - 1) tc5::commit(q_empty);  // the item's last QK: Q may be replaced
          if (jt > 0) ok = issue_pv(f - 1, jt == 1);
        }
        if (ok) issue_pv(t_glob + nkt - 1, nkt == 1);
      }
      __syncwarp();
    } else if (warp == 3) {
      // --------------------------------------------------------------------- V loads
      // each V tile is requested as soon as P.V has freed its stage
      bool ok = !*abort_flag;
      int nb0 = fetch_block(0), nb1 = fetch_block(1);
      for (int jt = 0; jt < nkt && ok; ++jt) {
        const int f = t_glob + jt;
        const int vs = f % C::VST;
        const int cur = nb0;
        nb0 = nb1;
        nb1 = fetch_block(jt + 2);
        if (f >= C::VST) ok = warp_wait(&v_empty[vs], (f / C::VST - 1) & 1, p.err, abort_flag);
        if (!ok) break;
        load_tile(true, jt, vs, cur);
      }
    } else if (warp == 2) {
      // ----------------------------------------------------------------- V release
      // Tile f is released after P.V of tile f - 1 was issued and completed (pv_done), which
      // also keeps vt_full at most one phase ahead of the MMA thread's waits; in an item's
      // last tile the rows of keys past the visible range are zeroed first.
      bool ok = !*abort_flag;
      for (int jt = 0; jt < nkt && ok; ++jt) {
        const int f = t_glob + jt;
        const int vs = f % C::VST;
        ok = warp_wait(&v_full[vs], (f / C::VST) & 1, p.err, abort_flag);
        if (ok && f >= 1) ok = pv_wait(f - 1);
        if (!ok) break;
        const int vis = kv_end - jt * C::BK;  // keys of this tile that some row sees
        if (vis < C::BK) {
          unsigned char* vbase = smem + C::OFF_V + vs * C::kKVBytes;
          const int n16 = (C::BK - vis) * 8 * HALVES;  // 16-byte chunks to clear
          for (int idx = lane; idx < n16; idx += 32) {
            const int hh = idx / ((C::BK - vis) * 8);
            const int rem = idx - hh * (C::BK - vis) * 8;
            *reinterpret_cast<uint4*>(vbase + hh * C::kBlk + (vis + (rem >> 3)) * 128 + ((rem & 7) << 4)) =
                make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(vt_full);
      }
    } else {
      // -------------------------------------------------------------------- softmax
      const int sw = warp - 4;  // TMEM lanes 32*sw .. 32*sw+31
      const int r = 32 * sw + lane;
      const int rt = r / G;          // position within the item
      const int rg = r - rt * G;     // q head within the group
      const bool live = rt < qrows;  // (rt < qrows implies r < G P)
      const int pos = pos0 + rt;
      const uint32_t trow = tmem + (static_cast<uint32_t>(32 * sw) << 16);
      float m_run = NEG_INF, l_run = 0.f;
      bool ok = !*abort_flag;
      for (int jt = 0; jt < nkt && ok; ++jt) {
        const int f = t_glob + jt;
        const int s = f & 1;
        ok = warp_wait(&s_full[s], (f >> 1) & 1, p.err, abort_flag);
        if (!ok) break;
        tc5::fence_after();
        float sc[128];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float v[32];
          tc5::ld32(trow + 128u * s + 32u * c, v);
#pragma unroll
          for (int x = 0; x < 32; ++x) sc[32 * c + x] = v[x];
        }
        tc5::wait_ld();
        tc5::fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_free[s]);
        // row max of the raw scores (qscale > 0 keeps the order, and fl(max * qscale) is the max
        // of the scaled scores), over eight independent partial maxima; the mask is a select
        // and only the diagonal tiles need it
        const int key0 = jt * C::BK;
        float mx8[8];
#pragma unroll
        for (int x = 0; x < 8; ++x) mx8[x] = NEG_INF;
        if (live && key0 + C::BK - 1 <= pos) {
#pragma unroll
          for (int c = 0; c < 128; ++c) mx8[c & 7] = fmaxf(mx8[c & 7], sc[c]);
        } else {
#pragma unroll
          for (int c = 0; c < 128; ++c) {
            sc[c] = (live && key0 + c <= pos) ? sc[c] : NEG_INF;
            mx8[c & 7] = fmaxf(mx8[c & 7], sc[c]);
          }
        }
        const float mraw = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                 fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
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
        // f32x2 pairs (two scores per instruction), four pairs of partial sums
        const float2 qs2 = make_float2(p.qscale, p.qscale);
        const float2 nb2 = make_float2(-base, -base);
        float2 ls4[4];
#pragma unroll
        for (int x = 0; x < 4; ++x) ls4[x] = make_float2(0.f, 0.f);
#pragma unroll
        for (int c = 0; c < 128; c += 2) {
          const float2 t = ffma2(make_float2(sc[c], sc[c + 1]), qs2, nb2);
          sc[c] = fast_exp2(t.x);
          sc[c + 1] = fast_exp2(t.y);
          ls4[(c >> 1) & 3] = fadd2(ls4[(c >> 1) & 3], make_float2(sc[c], sc[c + 1]));
        }
        const float2 ls2 = fadd2(fadd2(ls4[0], ls4[1]), fadd2(ls4[2], ls4[3]));
        const float lsum = ls2.x + ls2.y;
        l_run = l_run * corr + lsum;
        if (jt > 0 && __any_sync(0xffffffffu, resc)) {
          // O is rescaled only once every P.V issued so far has landed in it
          ok = pv_wait(f - 1);
          if (!ok) break;
          tc5::fence_after();
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            float o[32];
            tc5::ld32(trow + C::COL_O + 32u * c, o);
            tc5::wait_ld();
#pragma unroll
            for (int x = 0; x < 32; ++x) o[x] *= corr;
            tc5::st32(trow + C::COL_O + 32u * c, o);
          }
          tc5::wait_st();
        }
        if (f >= 2) {  // this P buffer was read by the P.V of tile f - 2
          ok = pv_wait(f - 2);
          if (!ok) break;
          tc5::fence_after();
        }
        // P row as bf16 pairs into TMEM, the A operand of P.V: column c holds keys 2c, 2c + 1
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          float pk[32];
#pragma unroll
          for (int x = 0; x < 32; ++x) pk[x] = __uint_as_float(pack_bf16x2(sc[64 * c + 2 * x], sc[64 * c + 2 * x + 1]));
          tc5::st32(trow + C::COL_P + 64u * (f & 1) + 32u * c, pk);
        }
        tc5::wait_st();
        tc5::fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[f & 1]);
      }
      if (ok) ok = pv_wait(t_glob + nkt - 1);
      if (ok) {
        tc5::fence_after();
        const float inv = live ? 1.f / l_run : 0.f;
        bf16* orow = p.out + static_cast<int64_t>(s0 + q0 + rt) * p.o_st + static_cast<int64_t>(h * G + rg) * p.o_sh;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          float o[32];
          tc5::ld32(trow + C::COL_O + 32u * c, o);
          tc5::wait_ld();
          if (live) {
#pragma unroll
            for (int x = 0; x < 4; ++x) {
              uint4 u;
              u.x = pack_bf16x2(o[8 * x + 0] * inv, o[8 * x + 1] * inv);
              u.y = pack_bf16x2(o[8 * x + 2] * inv, o[8 * x + 3] * inv);
              u.z = pack_bf16x2(o[8 * x + 4] * inv, o[8 * x + 5] * inv);
              u.w = pack_bf16x2(o[8 * x + 6] * inv, o[8 * x + 7] * inv);
              *reinterpret_cast<uint4*>(orow + 32 * c + 8 * x) = u;
            }
          }
        }
        tc5::fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(o_free);  // O is read: the next item's P.V may overwrite it
      }
    }
    t_glob += nkt;
    ++item_no;
  }
  __syncthreads();  // every role has finished its last item (the softmax warps read TMEM to the end)

  // teardown: no MMA may still be in flight when TMEM is released
  if (warp == 1) {
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
