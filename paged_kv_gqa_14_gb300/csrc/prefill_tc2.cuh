// Prefill-chunk attention on the 5th-generation tensor cores, two query tiles per CTA.
//
// Causal rule as everywhere ("mini_engine" README, "What it does": chunked prefill;
// "09 -- Mini Inference Engine (The Capstone)", "Week 3": mixed batches): row r of an n-row
// span sits at position ctx - n + r and sees keys 0 .. ctx - n + r.
//
// Item = (sequence, 2 P consecutive positions of its span, kv head h), P = floor(128 / G).
// It holds two 128-row query tiles: A = the first P positions, B = the next P, each stacking
// the G q heads that share kv head h (tile row r = position r / G of q head h G + r % G).
// Both tiles walk the same 128-key K/V tiles, so every K/V tile is staged once for 2 P
// positions x G heads; B sees at most one more key tile than A.
//
// Warp roles (11 warps):
//   warp 0      TMA producer: both Q tiles once per item (3-D map over q), then the K tiles
//               (one box per block of the tile and 64-dim half of kv head h) into a ring.
//   warp 1      allocates TMEM (512 columns: S_A, S_B 128 each, O_A, O_B d each) and, from one
//               thread, issues the tcgen05.mma of both tiles:
//                 S_X  = Q_X . K^T   (M 128, N 128, K d; both operands K-major in shared memory)
//                 O_X += P_X . V     (M 128, N d,  K 128; P_X from TMEM, V MN-major in shared)
//               in the order PV_A(j), QK_A(j+1), PV_B(j), QK_B(j+1), so each tile's product
//               chain QK -> softmax -> PV -> QK overlaps the other tile's.
//   warp 2      loads the V tiles into their own ring.  A V tile goes to the MMA on its own
//               TMA barrier, except an item's last tile: this warp first zeroes the rows of
//               keys past the visible range (0 * NaN would poison O) and then releases it.
//   warps 3-6   softmax of tile A, warps 7-10 softmax of tile B (warp w reads TMEM lanes
//               32 (w % 4) ..): thread = query row.  Loads its whole S row from TMEM into
//               registers with one wait, takes the row max, computes 2^(s scale - m) with
//               packed f32x2 FMA/add, keeps m and l in the log2 domain, writes P as bf16 pairs
//               over the first 64 columns of its own S (the next S = Q K^T of that tile is
//               issued only after this P.V has completed, so the alias is safe), and rescales
//               O in TMEM only when the row max grows by more than 2^8.  At the end it reads O,
//               divides by l and stores bf16.
// Every wait is bounded; a CTA that times out sets PKV_DEVERR_TIMEOUT and finishes its items
// without further work.
#pragma once

#include <cuda.h>

#include "decode_tc.cuh"
#include "prefill.cuh"
#include "tcgen05.cuh"

namespace pkv {

struct PrefillTc2Params {
  CUtensorMap tmap_q;  // 3-D {d, Hq, T}, box {64, G, P}, 128B swizzle
  CUtensorMap tmap_k;  // 4-D {d, Hkv, block_size, num_blocks}, box {64, 1, block_size, 1}, 128B swizzle
  CUtensorMap tmap_v;
  PrefillParams p;
  int group;  // G = Hq / Hkv
  int prows;  // P = floor(128 / G): positions per query tile
};

template <int D>
struct PrefillTc2Cfg {
  static constexpr int kThreads = 352;
  static constexpr int BQ = 128;  // rows per query tile
  static constexpr int BK = 128;  // keys per K/V tile
  static constexpr int HALVES = D / 64;
  static constexpr int kBlk = 128 * 128;  // one [128 rows][64 elements] swizzled block: 16 KB
  static constexpr int kQBytes = BQ * D * 2;
  static constexpr int kKVBytes = BK * D * 2;
  static constexpr int KST = D == 128 ? 2 : 3;  // (d 128: Q 64 KB + K 2 x 32 KB + V 2 x 32 KB)
  static constexpr int VST = D == 128 ? 2 : 3;
  static constexpr int OFF_Q = 0;  // Q_A, Q_B
  static constexpr int OFF_K = OFF_Q + 2 * kQBytes;
  static constexpr int OFF_V = OFF_K + KST * kKVBytes;
  static constexpr int OFF_BAR = OFF_V + VST * kKVBytes;
  static constexpr int OFF_XCH = OFF_BAR + 256;  // row max / sum exchange: [2 halves][4][2][32] floats
  static constexpr int kSmemBytes = OFF_XCH + 2048 + 1024;  // + alignment slack
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t COL_S0 = 0;    // S_X at 128 X; P_X over its first 64 columns
  static constexpr uint32_t COL_O0 = 256;  // O_X at 256 + 128 X
  static_assert(D <= 128, "TMEM columns: 2 x S 128 + 2 x O 128");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

// Two fp32 lanes per instruction (packed f32x2, Blackwell).
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

template <int D>
__global__ void __launch_bounds__(352, 1) prefill_tc2_kernel(const __grid_constant__ PrefillTc2Params P) {
  using C = PrefillTc2Cfg<D>;
  constexpr int HALVES = C::HALVES;
  const PrefillParams& p = P.p;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars + 0;
  uint64_t* k_full = bars + 1;    // [KST]
  uint64_t* k_empty = bars + 4;   // [KST] both QK of the tile completed
  uint64_t* v_full = bars + 7;    // [VST] TMA landed
  uint64_t* v_empty = bars + 10;  // [VST] both PV of the tile completed
  uint64_t* v_zero = bars + 13;   // an item's last V tile: rows past the visible range zeroed
  uint64_t* s_full = bars + 14;   // [2] S_X written
  uint64_t* p_full = bars + 16;   // [2] P_X written (8 warps)
  uint64_t* pv_done = bars + 18;  // [2] P_X . V completed
  uint64_t* fin = bars + 20;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 21);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 22);
  uint64_t* xbar = bars + 24;     // [4] softmax warp pair on SM sub-partition q exchanged its values
  float* xch = reinterpret_cast<float*>(smem + C::OFF_XCH);
  static_assert(C::KST <= 3 && C::VST <= 3, "barrier layout");
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
    mbar_init(v_zero, 1);
    for (int x = 0; x < 2; ++x) {
      mbar_init(&s_full[x], 1);
      mbar_init(&p_full[x], 8);
      mbar_init(&pv_done[x], 1);
    }
    mbar_init(fin, 1);
    for (int q = 0; q < 4; ++q) mbar_init(&xbar[q], 2);
    fence_mbar_init();
    *abort_flag = 0;
  }
  if (warp == 0 && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&P.tmap_q)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&P.tmap_k)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&P.tmap_v)) : "memory");
  }
  // TMEM is taken while the planner still runs (programmatic dependent launch)
  if (warp == 1) {
    tc5::alloc(tmem_slot, C::TMEM_COLS);
    tc5::relinquish();
  }
  tc5::fence_before();
  __syncthreads();
  tc5::fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();  // the tile list is written by the planner kernel
  pdl_trigger();
  const int n_tiles = p.plan.header[3];
  const int total = n_tiles * p.hkv;
  const int nact = min(max(p.plan.header[5], 0), static_cast<int>(gridDim.x));
  if (static_cast<int>(blockIdx.x) >= total || static_cast<int>(blockIdx.x) >= nact) {
    if (warp == 1) tc5::dealloc(tmem, C::TMEM_COLS);
    return;
  }
  const int G = P.group;
  const int PR = P.prows;
  const uint64_t pol = l2_policy_evict_last();  // K/V tiles are re-read by the other items

  int t_glob = 0;          // K/V tiles this CTA has processed (ring slots)
  int issued = 0;          // K (warp 0) or V (warp 2) tiles this warp has requested
  int cnt0 = 0, cnt1 = 0;  // per query tile: S/P/PV rounds so far (barrier phases)
  int xuse = 0;            // softmax: row max / sum exchanges so far (xbar phase, buffer)
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
    const int q0 = j * 2 * PR;
    const int rows0 = min(PR, n - q0);               // positions of tile A
    const int rows1 = max(0, min(PR, n - q0 - PR));  // positions of tile B (0: empty)
    const int pos0 = ctx - n + q0;
    const int nk0 = ceil_div(pos0 + rows0, C::BK);   // key tiles of each query tile
    const int nk1 = rows1 > 0 ? ceil_div(pos0 + PR + rows1, C::BK) : 0;
    const int kv_end = rows1 > 0 ? pos0 + PR + rows1 : pos0 + rows0;  // keys [0, kv_end) are used
    const int nkt = max(nk0, nk1);

    // One K or V tile of 128 keys, issued by one warp: 128 / bs boxes of one whole block of kv
    // head h per 64-dim half, lane = box x half.  Boxes past kv_end are not loaded.  Block ids
    // are read two tiles ahead of their use.
    const int bs = 1 << p.bs_log2;
    const int lbox = lane / HALVES;
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
      bool ok = !*abort_flag;
      if (ok) {
        const int nq = rows1 > 0 ? 2 : 1;
        if (lane == 0) mbar_arrive_expect_tx(q_full, static_cast<uint32_t>(nq * HALVES * G * PR * 128));
        __syncwarp();
        if (lane < nq * HALVES) {
          const int x = lane / HALVES, hh = lane - x * HALVES;
          tma_load_3d(smem + C::OFF_Q + x * C::kQBytes + hh * C::kBlk, &P.tmap_q, hh * 64, h * G, s0 + q0 + x * PR,
                      q_full);
        }
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
        ++issued;
      }
    } else if (warp == 1) {
      // ------------------------------------------------------------------- MMA issuer
      if (lane == 0) {
        constexpr uint32_t kIdescQK = tc5::idesc_bf16_f32(128, 128);
        constexpr uint32_t kIdescPV = tc5::idesc_bf16_f32(128, D, true);
        bool ok = wait_or_abort(q_full, item_no & 1, p.err, abort_flag);
        int c0 = cnt0, c1 = cnt1;  // rounds issued per query tile
        int k_waited = -1, v_waited = -1;
        auto wait_k = [&](int jt) -> bool {
          if (k_waited >= jt) return true;
          k_waited = jt;
          const int f = t_glob + jt;
          if (!wait_or_abort(&k_full[f % C::KST], (f / C::KST) & 1, p.err, abort_flag)) return false;
          tc5::fence_after();
          return true;
        };
        auto wait_v = [&](int jt) -> bool {
          if (v_waited >= jt) return true;
          v_waited = jt;
          const int f = t_glob + jt;
          const bool last = jt == nkt - 1;
          if (!(last ? wait_or_abort(v_zero, item_no & 1, p.err, abort_flag)
                     : wait_or_abort(&v_full[f % C::VST], (f / C::VST) & 1, p.err, abort_flag)))
            return false;
          tc5::fence_after();
          return true;
        };
        auto qk = [&](int x, int jt) -> bool {
          if (!wait_k(jt)) return false;
          const int ks = (t_glob + jt) % C::KST;
          const uint32_t qb = sb + C::OFF_Q + x * C::kQBytes;
          const uint32_t kb = sb + C::OFF_K + ks * C::kKVBytes;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * C::kBlk + (kk & 3) * 32;
            tc5::mma_ss(tmem + C::COL_S0 + 128u * x, tc5::smem_desc_k128(qb + off), tc5::smem_desc_k128(kb + off),
                        kIdescQK, kk > 0 ? 1u : 0u);
          }
          tc5::commit(&s_full[x]);
          return true;
        };
        auto pv = [&](int x, int jt) -> bool {
          if (!wait_v(jt)) return false;
          if (!wait_or_abort(&p_full[x], (x ? c1 : c0) & 1, p.err, abort_flag)) return false;
          tc5::fence_after();
          const uint32_t vst = sb + C::OFF_V + ((t_glob + jt) % C::VST) * C::kKVBytes;
#pragma unroll
          for (int kk = 0; kk < C::BK / 16; ++kk)  // A = P_X from TMEM: 16 keys = 8 columns
            tc5::mma_ts(tmem + C::COL_O0 + 128u * x, tmem + C::COL_S0 + 128u * x + 8u * kk,
                        tc5::smem_desc_mn128(vst + kk * 2048, C::kBlk), kIdescPV, (jt == 0 && kk == 0) ? 0u : 1u);
          tc5::commit(&pv_done[x]);
          return true;
        };
        // round 0: S of both tiles
        if (ok) ok = qk(0, 0);
        if (ok && nk1 > 0) ok = qk(1, 0);
        if (ok) tc5::commit(&k_empty[t_glob % C::KST]);
        for (int jt = 0; jt < nkt && ok; ++jt) {
#pragma unroll
          for (int x = 0; x < 2; ++x) {
            const int nkx = x ? nk1 : nk0;
            if (!ok || jt >= nkx) continue;
            int& cx = x ? c1 : c0;
            ok = pv(x, jt);
            if (ok && jt + 1 < nkx) {
              // S_X of the next tile overwrites P_X: wait until this P.V has read it
              ok = wait_or_abort(&pv_done[x], cx & 1, p.err, abort_flag);
              if (ok) {
                tc5::fence_after();
                ok = qk(x, jt + 1);
              }
            }
            ++cx;
          }
          if (!ok) break;
          tc5::commit(&v_empty[(t_glob + jt) % C::VST]);
          if (jt + 1 < nkt) tc5::commit(&k_empty[(t_glob + jt + 1) % C::KST]);
        }
      }
      __syncwarp();
    } else if (warp == 2) {
      // --------------------------------------------------------------------- V loads
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
        ++issued;
        if (jt == nkt - 1) {
          // the item's last tile: zero the rows of keys past the visible range, then release
          ok = warp_wait(&v_full[vs], (f / C::VST) & 1, p.err, abort_flag);
          if (!ok) break;
          const int vis = kv_end - jt * C::BK;
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
          if (lane == 0) mbar_arrive(v_zero);
        }
      }
    } else {
      // -------------------------------------------------------------------- softmax
      // The two warps on each SM sub-partition (warps w and w + 4) share TMEM lanes
      // 32 (w % 4) .. + 31, i.e. 32 query rows: warp half hh takes key columns
      // [64 hh, 64 hh + 64) of every S tile, first of tile A, then of tile B.  Row max and row
      // sum are combined through shared memory (an mbarrier per warp pair).
      const int sw = warp & 3;
      const int hh = (warp - 3) >> 2;  // 0: warps 3-6, 1: warps 7-10
      const int r = 32 * sw + lane;
      const int rt = r / G;  // position within a query tile
      const int rg = r - rt * G;
      const uint32_t trow = tmem + (static_cast<uint32_t>(32 * sw) << 16);
      float* xmine = xch + (hh * 4 + sw) * 64;           // [parity][lane] of this warp
      const float* xother = xch + ((1 - hh) * 4 + sw) * 64;
      // the partner warp's value of this row; both warps arrive on the pair's mbarrier after
      // writing (release) and read after its phase completes (acquire).  Bounded: false on
      // a timeout or an abort, like every other wait.
      auto exchange = [&](float v, float& other) -> bool {
        const int u = xuse++;
        xmine[(u & 1) * 32 + lane] = v;
        __syncwarp();
        if (lane == 0) mbar_arrive(&xbar[sw]);
        if (!warp_wait(&xbar[sw], u & 1, p.err, abort_flag)) return false;
        other = xother[(u & 1) * 32 + lane];
        return true;
      };
      float m_run[2] = {NEG_INF, NEG_INF}, l_run[2] = {0.f, 0.f};
      int c[2] = {cnt0, cnt1};
      bool ok = !*abort_flag;
      for (int jt = 0; jt < nkt && ok; ++jt) {
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          const int nk_x = x ? nk1 : nk0;
          if (!ok || jt >= nk_x) continue;
          const bool live = rt < (x ? rows1 : rows0);  // (rt < rows implies r < G P)
          const int pos = pos0 + x * PR + rt;
          const uint32_t t_s = trow + C::COL_S0 + 128u * x;
          const uint32_t t_o = trow + C::COL_O0 + 128u * x;
          ok = warp_wait(&s_full[x], c[x] & 1, p.err, abort_flag);
          if (!ok) break;
          tc5::fence_after();
          const int key0 = jt * C::BK + 64 * hh;  // this warp's first key
          // the warp's rows see all 64 of its keys: no mask (warp-uniform)
          const bool full = __all_sync(0xffffffffu, live && key0 + 63 <= pos);
          float sc[64];
          tc5::ld32(t_s + 64u * hh, *reinterpret_cast<float(*)[32]>(sc));
          tc5::ld32(t_s + 64u * hh + 32u, *reinterpret_cast<float(*)[32]>(sc + 32));
          tc5::wait_ld();
          if (!full) {  // masked keys -> -inf
#pragma unroll
            for (int i = 0; i < 64; ++i) sc[i] = (live && key0 + i <= pos) ? sc[i] : NEG_INF;
          }
          float mx8[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) mx8[i] = NEG_INF;
#pragma unroll
          for (int i = 0; i < 64; ++i) mx8[i & 7] = fmaxf(mx8[i & 7], sc[i]);
          float mraw = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                             fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
          // both halves of the row are in registers after this barrier, so P may now be
          // written over S's first 64 columns (which hold half 0's scores)
          float mpart;
          ok = exchange(mraw, mpart);
          if (!ok) break;
          mraw = fmaxf(mraw, mpart);
          const float mx = mraw * p.qscale;  // the row max (qscale > 0 keeps the order); -inf stays -inf
          float corr = 1.f;
          bool resc = false;
          if (m_run[x] == NEG_INF) {
            m_run[x] = mx;
          } else if (mx > m_run[x] + 8.f) {
            corr = fast_exp2(m_run[x] - mx);
            m_run[x] = mx;
            resc = true;
          }
          const float base = m_run[x] == NEG_INF ? 0.f : m_run[x];
          if (jt > 0 && __any_sync(0xffffffffu, resc)) {
            // O is rescaled (this warp's half of its columns) once the previous P.V landed
            ok = warp_wait(&pv_done[x], (c[x] - 1) & 1, p.err, abort_flag);
            if (!ok) break;
            tc5::fence_after();
#pragma unroll 1
            for (int ch = 0; ch < D / 64; ++ch) {
              const uint32_t col = t_o + static_cast<uint32_t>(hh * (D / 2) + 32 * ch);
              float o[32];
              tc5::ld32(col, o);
              tc5::wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i) o[i] *= corr;
              tc5::st32(col, o);
            }
            tc5::wait_st();
          }
          // p = 2^(s qscale - base) with packed f32x2 FMA/add; P as bf16 pairs: keys
          // 64 hh + 2 j, + 1 in column 32 hh + j
          const float2 qs2 = make_float2(p.qscale, p.qscale);
          const float2 nb2 = make_float2(-base, -base);
          float2 ls4[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) ls4[i] = make_float2(0.f, 0.f);
#pragma unroll
          for (int ch = 0; ch < 2; ++ch) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              const float2 t = ffma2(make_float2(sc[32 * ch + i], sc[32 * ch + i + 1]), qs2, nb2);
              const float2 e = make_float2(fast_exp2(t.x), fast_exp2(t.y));  // 2^-inf = 0
              ls4[(i >> 1) & 3] = fadd2(ls4[(i >> 1) & 3], e);
              pk[i >> 1] = pack_bf16x2(e.x, e.y);
            }
            tc5::st16(t_s + 32u * hh + 16u * ch, pk);
          }
          const float2 ls = fadd2(fadd2(ls4[0], ls4[1]), fadd2(ls4[2], ls4[3]));
          l_run[x] = l_run[x] * corr + (ls.x + ls.y);  // this half's share of the row sum
          tc5::wait_st();
          tc5::fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&p_full[x]);
          ++c[x];
        }
      }
      // epilogue per query tile: full row sum, O / l, bf16 store of this warp's half of d
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        const int nk_x = x ? nk1 : nk0;
        if (nk_x == 0) continue;
        if (ok) ok = warp_wait(&pv_done[x], (c[x] - 1) & 1, p.err, abort_flag);
        if (!ok) break;
        tc5::fence_after();
        const bool live = rt < (x ? rows1 : rows0);
        float lpart;
        ok = exchange(l_run[x], lpart);
        if (!ok) break;
        const float l = l_run[x] + lpart;
        const float inv = live ? 1.f / l : 0.f;
        const uint32_t t_o = trow + C::COL_O0 + 128u * x;
        bf16* orow = p.out + static_cast<int64_t>(s0 + q0 + x * PR + rt) * p.o_st +
                     static_cast<int64_t>(h * G + rg) * p.o_sh + hh * (D / 2);
#pragma unroll 1
        for (int ch = 0; ch < D / 64; ++ch) {
          float o[32];
          tc5::ld32(t_o + static_cast<uint32_t>(hh * (D / 2) + 32 * ch), o);
          tc5::wait_ld();
          if (live) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              uint4 u;
              u.x = pack_bf16x2(o[8 * i + 0] * inv, o[8 * i + 1] * inv);
              u.y = pack_bf16x2(o[8 * i + 2] * inv, o[8 * i + 3] * inv);
              u.z = pack_bf16x2(o[8 * i + 4] * inv, o[8 * i + 5] * inv);
              u.w = pack_bf16x2(o[8 * i + 6] * inv, o[8 * i + 7] * inv);
              *reinterpret_cast<uint4*>(orow + 32 * ch + 8 * i) = u;
            }
          }
        }
        tc5::fence_before();
      }
    }
    t_glob += nkt;
    cnt0 += nk0;
    cnt1 += nk1;
    ++item_no;
    __syncthreads();  // the item's buffers (Q, S, O, P) are free for the next item
  }

  // teardown: no copy may still be landing in shared memory when the CTA leaves (after an
  // abort a load may be unconsumed: wait, bounded, for the last fill of each stage) ...
  if (warp == 0 || warp == 2) {
    const int st = warp == 0 ? C::KST : C::VST;
    uint64_t* full = warp == 0 ? k_full : v_full;
    for (int f = max(0, issued - st); f < issued; ++f) mbar_wait(&full[f % st], (f / st) & 1, p.err);
  }
  // ... and no MMA may still be in flight when TMEM is released
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
