// Fused RoPE + KV-cache append ("mini_engine" README, "Next: fused kernels": fused RoPE
// and fused QKV split + KV-cache write; "09 -- Mini Inference Engine (The Capstone)",
// "Week 4 -- Paged KV cache": pool of fixed-size blocks addressed by slot; the block size is
// 16 by default and any power of two from 8 to 128 here).
//
// One warp per new token, four tokens per CTA, no CTA-wide barrier.  A warp first issues the
// loads of its token's q, k and v rows (their addresses do not depend on the position) and of
// its position and slot, then computes the d/2 rotation angles into a warp-private table in
// shared memory: angle = pos * f_i with f_i = theta^(-2i/d) (fp64 on the host), taken modulo
// one turn exactly in 64-bit integer arithmetic (RopeFreqs), split exactly into a quarter turn
// and a remainder in [-pi/4, pi/4) that reaches fp32 with one rounding, then sincosf in fp32
// and an exact quarter-turn swap.  Every head of q (in place) and k (into the slot) is
// rotated pairwise (i, i + d/2) in fp32 and rounded to bf16 nearest-even; v is a 16-byte
// vector copy.  All global accesses are 16-byte vectors along head_dim; the lanes of a warp
// cover consecutive 16-byte chunks of a head row, so every access is coalesced.
//
// Error of a rotated fp32 value before its bf16 rounding, for a pair (x, y) at a position
// below 2^31: the fp32 remainder angle is within 2^-25 rad of the exact one (one rounding at
// |r| < 1), plus pos * 2 pi / 2^64 from the rounding of F_i; sincosf is within 2 ulp (2^-23)
// of sin and cos; the two products and the difference add at most 2^-23 (|x| + |y|).  In
// all, |error| <= 2.7e-7 (|x| + |y|), below 2^-21 (|x| + |y|).
#include <math.h>

#include <cmath>

#include "common.cuh"
#include "internal.h"

namespace pkv {
namespace {

constexpr int kAppendWarps = 4;  // warps per CTA
// Warps per token (each computes the whole angle table, so they never synchronise).  Measured
// on GB300 on the 2248-token mixed step: one warp 10.5 us, two warps 10.5-10.9 us, one CTA of
// two warps per token with a CTA barrier 10.8 us.
constexpr int kWarpsPerToken = 1;

// Where each token's position and slot come from: explicit arrays, or (qsl != nullptr)
// derived on the device from the scheduler's tables.
struct AppendSrc {
  const int64_t* positions;
  const int64_t* slots;
  const int32_t* qsl;
  const int32_t* ctxl;
  const int32_t* bt;
  int64_t bt_stride, max_blocks, num_seqs;
  int bs_log2;  // log2 of the pool's block size
  int64_t* pos_out;
  int64_t* slot_out;
};

// The rotation frequencies as fractions of a turn in 0.64 fixed point:
// F_i = round(frac(f_i / (2 pi)) * 2^64), f_i = theta^(-2i/d).  The angle of position p is
// then p f_i = 2 pi (p F_i / 2^64) modulo whole turns, and its part modulo one turn is the
// low 64 bits of the integer product p F_i: exact up to the rounding of F_i (at most p / 2^64
// of a turn), with no floating-point range reduction.
struct RopeFreqs {
  unsigned long long F[kMaxHeadDim / 2];
};

// 2 pi / 2^32 (radians per unit of the top 32 bits of a 0.64 fixed-point turn) as the sum of
// two floats: hi the float nearest to it, lo the float nearest to the rest.
constexpr float kTwoPiOver2p32Hi = 1.4629180792671596e-09f;
constexpr float kTwoPiOver2p32Lo =
    static_cast<float>(1.4629180792671596e-09 - static_cast<double>(kTwoPiOver2p32Hi));

// cos and sin of the angle 2 pi turn / 2^64.  The nearest quarter turn k = round(4 turn / 2^64)
// mod 4 and the remainder rem = turn - k 2^62, a signed integer in [-2^61, 2^61], are exact;
// r = 2 pi rem / 2^64 in [-pi/4, pi/4] is formed from rem's top word (rounded to a float, the
// rounding kept as a small exact integer), its low word and the two-float constant, with one
// fp32 rounding in the last step.  (cos, sin) of k pi/2 + r are (cos r, sin r) turned by k
// quarter turns: a swap and sign changes, exact.
__device__ __forceinline__ float2 cos_sin_of_turn(unsigned long long turn) {
  const unsigned k = static_cast<unsigned>((turn + (1ull << 61)) >> 62);  // 0..3, wraps mod 4
  const long long rem = static_cast<long long>(turn - (static_cast<unsigned long long>(k) << 62));
  const int hi = static_cast<int>(rem >> 32);  // |hi| <= 2^29
  const unsigned lo = static_cast<unsigned>(rem);
  const float hi_f = static_cast<float>(hi);
  const int hi_rest = hi - static_cast<int>(hi_f);  // exact, |hi_rest| <= 16
  const float x_lo = fmaf(static_cast<float>(lo), 2.3283064365386963e-10f /* 2^-32 */, static_cast<float>(hi_rest));
  const float r = fmaf(hi_f, kTwoPiOver2p32Hi, fmaf(hi_f, kTwoPiOver2p32Lo, x_lo * kTwoPiOver2p32Hi));
  float s, c;
  sincosf(r, &s, &c);
  switch (k & 3u) {
    case 0: return make_float2(c, s);
    case 1: return make_float2(-s, c);
    case 2: return make_float2(-c, -s);
    default: return make_float2(s, -c);
  }
}

template <typename CS>
__device__ __forceinline__ void rotate8(uint4& lo, uint4& hi, const CS& cs) {
  uint32_t* a = reinterpret_cast<uint32_t*>(&lo);
  uint32_t* b = reinterpret_cast<uint32_t*>(&hi);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float2 c0 = cs[2 * j], c1 = cs[2 * j + 1];
    const float x0 = bf16lo(a[j]), x1 = bf16hi(a[j]);  // first half, pairs 2j, 2j+1
    const float y0 = bf16lo(b[j]), y1 = bf16hi(b[j]);  // second half, same pairs
    a[j] = pack_bf16x2(x0 * c0.x - y0 * c0.y, x1 * c1.x - y1 * c1.y);
    b[j] = pack_bf16x2(y0 * c0.x + x0 * c0.y, y1 * c1.x + x1 * c1.y);
  }
}

// Position and slot of token t, derived on the device from the scheduler's tables: the
// token's sequence b is the last one with query_start_loc[b] <= t (found by a warp-wide
// search, 32 samples per round), it sits at position ctx_b - n_b + (t - qsl[b]) and its slot
// is row pos % bs of block block_tables[b][pos / bs].  Tokens outside every span get slot -1.
__device__ __forceinline__ void derive_slot(const AppendSrc& src, int64_t t, int lane, int64_t num_blocks, unsigned int* err,
                            int64_t& pos, int64_t& slot) {
  const int32_t* qsl = src.qsl;
  int lo = 0, hi = static_cast<int>(src.num_seqs);  // inclusive range of qsl indices
  int b = -1;
  for (int round = 0; round < 8; ++round) {  // 32^8 covers any int32 count
    const int len = hi - lo + 1;
    if (len <= 32) {
      const int idx = lo + lane;
      const unsigned m = __ballot_sync(0xffffffffu, idx <= hi && qsl[idx] <= t);
      b = lo + __popc(m) - 1;
      break;
    }
    const int stride = (len + 31) / 32;
    const int idx = lo + lane * stride;  // samples past hi take no part in the count
    const unsigned m = __ballot_sync(0xffffffffu, idx <= hi && qsl[idx] <= t);
    const int k = __popc(m) - 1;
    if (k < 0) break;
    const int nlo = lo + k * stride;
    hi = min(hi, nlo + stride - 1);
    lo = nlo;
  }
  pos = 0;
  slot = -1;
  if (b < 0 || b >= src.num_seqs) return;  // before the first or after the last span
  const int s0 = qsl[b];
  const int n = qsl[b + 1] - s0;
  const int ctx = src.ctxl[b];
  if (n <= 0 || t - s0 >= n) return;
  if (ctx < n) {
    if (lane == 0) raise_error(err, PKV_DEVERR_SPAN);
    return;
  }
  pos = static_cast<int64_t>(ctx) - n + (t - s0);
  const int64_t page = pos >> src.bs_log2;
  if (page >= src.max_blocks) {
    if (lane == 0) raise_error(err, PKV_DEVERR_CONTEXT);
    return;
  }
  const int blk = src.bt[static_cast<int64_t>(b) * src.bt_stride + page];
  if (blk < 0 || blk >= num_blocks) {
    if (lane == 0) raise_error(err, PKV_DEVERR_BLOCK_RANGE);
    return;
  }
  slot = (static_cast<int64_t>(blk) << src.bs_log2) + (pos & ((int64_t(1) << src.bs_log2) - 1));
}

// Row items a lane holds in registers from the start (a q or k item is one 16-byte chunk pair
// (i, i + d/2) of a head, a v item one 16-byte chunk); items past these counts are read later.
constexpr int kQPrefetch = 4 / kWarpsPerToken;  // q items per lane: 16 q heads at d 128 have 128
constexpr int kKPrefetch = 2 / kWarpsPerToken;  // k items per lane: 8 kv heads at d 128 have 64
constexpr int kVPrefetch = 4 / kWarpsPerToken;  // v items per lane: 8 kv heads at d 128 have 128

template <int D>
__global__ void __launch_bounds__(kAppendWarps * 32) kv_append_kernel(
    bf16* __restrict__ q, int64_t q_st, int64_t q_sh, const bf16* __restrict__ k, int64_t k_st,
    int64_t k_sh, const bf16* __restrict__ v, int64_t v_st, int64_t v_sh, const __grid_constant__ AppendSrc src,
    bf16* __restrict__ k_cache, bf16* __restrict__ v_cache, int64_t num_tokens, int64_t num_slots, int hq, int hkv,
    const __grid_constant__ RopeFreqs fr, unsigned int* err) {
  constexpr int HALF = D / 2;
  constexpr int CH = HALF / 8;  // 16-byte chunks per half head
  constexpr int VCH = D / 8;    // 16-byte chunks per v head
  __shared__ float2 cs_all[kAppendWarps][HALF];

  pdl_wait();  // q, k, v and the index inputs may come from the previous kernel
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int kTokensPerCta = kAppendWarps / kWarpsPerToken;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * kTokensPerCta + warp / kWarpsPerToken;
  const int sub = warp % kWarpsPerToken;  // this warp takes items sub, sub + W, ... (W = warps per token)
  constexpr int kStride = 32 * kWarpsPerToken;
  if (t >= num_tokens) return;  // warp-uniform; nothing below synchronises more than the warp
  float2* cs = cs_all[warp];
  const int nq = hq * CH, nk = hkv * CH, nv = hkv * VCH;
  auto q_row = [&](int item, int& c) -> bf16* {
    const int head = item / CH;
    c = item - head * CH;
    return q + t * q_st + head * q_sh;
  };
  auto k_row = [&](int item, int& c) -> const bf16* {
    const int head = item / CH;
    c = item - head * CH;
    return k + t * k_st + head * k_sh;
  };
  // position and slot first (explicit arrays: one load each, lane 0)
  int64_t pos = 0, slot = -1;
  if (!src.qsl && lane == 0) {
    pos = src.positions[t];
    slot = src.slots[t];
  }
  // the token's rows
  uint4 qlo[kQPrefetch], qhi[kQPrefetch], klo[kKPrefetch], khi[kKPrefetch], vx[kVPrefetch];
#pragma unroll
  for (int j = 0; j < kQPrefetch; ++j) {
    const int item = lane + 32 * sub + kStride * j;
    if (item < nq) {
      int c;
      const bf16* row = q_row(item, c);
      qlo[j] = *reinterpret_cast<const uint4*>(row + c * 8);
      qhi[j] = *reinterpret_cast<const uint4*>(row + HALF + c * 8);
    }
  }
#pragma unroll
  for (int j = 0; j < kKPrefetch; ++j) {
    const int item = lane + 32 * sub + kStride * j;
    if (item < nk) {
      int c;
      const bf16* row = k_row(item, c);
      klo[j] = *reinterpret_cast<const uint4*>(row + c * 8);
      khi[j] = *reinterpret_cast<const uint4*>(row + HALF + c * 8);
    }
  }
#pragma unroll
  for (int j = 0; j < kVPrefetch; ++j) {
    const int item = lane + 32 * sub + kStride * j;
    if (item < nv) {
      const int h = item / VCH, c = item - (item / VCH) * VCH;
      vx[j] = *reinterpret_cast<const uint4*>(v + t * v_st + h * v_sh + c * 8);
    }
  }
  if (src.qsl) {
    derive_slot(src, t, lane, num_slots >> src.bs_log2, err, pos, slot);
  } else {
    pos = __shfl_sync(0xffffffffu, pos, 0);
    slot = __shfl_sync(0xffffffffu, slot, 0);
  }
  if (lane == 0 && sub == 0) {
    if (src.pos_out) src.pos_out[t] = pos;
    if (src.slot_out) src.slot_out[t] = slot;
  }

  // the token's angles modulo one turn: pos F_i mod 2^64 in 0.64 fixed point
  for (int i = lane; i < HALF; i += 32) cs[i] = cos_sin_of_turn(static_cast<unsigned long long>(pos) * fr.F[i]);
  const bool in_range = slot < num_slots;
  const bool write_kv = slot >= 0 && in_range;
  if (!in_range && lane == 0 && sub == 0) raise_error(err, PKV_DEVERR_SLOT_RANGE);
  __syncwarp();
  // every item of this lane is chunk c = lane % CH of some head (32 is a multiple of CH): its
  // eight (cos, sin) pairs are held in registers
  float2 my_cs[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) my_cs[i] = cs[(lane % CH) * 8 + i];

  // q heads rotated in place
#pragma unroll
  for (int j = 0; j < kQPrefetch; ++j) {
    const int item = lane + 32 * sub + kStride * j;
    if (item < nq) {
      int c;
      bf16* row = q_row(item, c);
      rotate8(qlo[j], qhi[j], my_cs);
      *reinterpret_cast<uint4*>(row + c * 8) = qlo[j];
      *reinterpret_cast<uint4*>(row + HALF + c * 8) = qhi[j];
    }
  }
  for (int item = lane + 32 * sub + kStride * kQPrefetch; item < nq; item += kStride) {
    int c;
    bf16* row = q_row(item, c);
    uint4 lo = *reinterpret_cast<const uint4*>(row + c * 8);
    uint4 hi = *reinterpret_cast<const uint4*>(row + HALF + c * 8);
    rotate8(lo, hi, my_cs);
    *reinterpret_cast<uint4*>(row + c * 8) = lo;
    *reinterpret_cast<uint4*>(row + HALF + c * 8) = hi;
  }
  if (!write_kv) return;
  // k heads rotated into the cache row of `slot`, v heads copied there
#pragma unroll
  for (int j = 0; j < kKPrefetch; ++j) {
    const int item = lane + 32 * sub + kStride * j;
    if (item < nk) {
      const int h = item / CH, c = item - (item / CH) * CH;
      rotate8(klo[j], khi[j], my_cs);
      bf16* dst = k_cache + (slot * hkv + h) * D;
      *reinterpret_cast<uint4*>(dst + c * 8) = klo[j];
      *reinterpret_cast<uint4*>(dst + HALF + c * 8) = khi[j];
    }
  }
  for (int item = lane + 32 * sub + kStride * kKPrefetch; item < nk; item += kStride) {
    int c;
    const bf16* row = k_row(item, c);
    const int h = item / CH;
    uint4 lo = *reinterpret_cast<const uint4*>(row + c * 8);
    uint4 hi = *reinterpret_cast<const uint4*>(row + HALF + c * 8);
    rotate8(lo, hi, my_cs);
    bf16* dst = k_cache + (slot * hkv + h) * D;
    *reinterpret_cast<uint4*>(dst + c * 8) = lo;
    *reinterpret_cast<uint4*>(dst + HALF + c * 8) = hi;
  }
#pragma unroll
  for (int j = 0; j < kVPrefetch; ++j) {
    const int item = lane + 32 * sub + kStride * j;
    if (item < nv) {
      const int h = item / VCH, c = item - (item / VCH) * VCH;
      *reinterpret_cast<uint4*>(v_cache + (slot * hkv + h) * D + c * 8) = vx[j];
    }
  }
  for (int item = lane + 32 * sub + kStride * kVPrefetch; item < nv; item += kStride) {
    const int h = item / VCH, c = item - (item / VCH) * VCH;
    *reinterpret_cast<uint4*>(v_cache + (slot * hkv + h) * D + c * 8) =
        *reinterpret_cast<const uint4*>(v + t * v_st + h * v_sh + c * 8);
  }
}

}  // namespace

namespace {

// round(frac(f / (2 pi)) * 2^64) for f > 0, to within one unit: 2^64 / (2 pi) is a double-double
// (kHi + kLo), the product's rounding error is recovered by an FMA, and whole turns drop out
// modulo 2^64 through an exact fmod, so f above one turn per position (rope_theta < 1) is
// reduced as exactly as f below.  False when f * 2^64 / (2 pi) is not finite.
bool turn_fraction_0p64(double f, unsigned long long* out) {
  constexpr double kHi = 2.9358905032820014e+18;  // 2^64 / (2 pi) = kHi + kLo
  constexpr double kLo = -181.50375616818445;
  constexpr double kTwo64 = 18446744073709551616.0;
  const double p = f * kHi;
  if (!std::isfinite(p) || !(f >= 0.0)) return false;
  const double e = fma(f, kHi, -p) + f * kLo;  // f (kHi + kLo) - p
  const double pm = fmod(p, kTwo64);           // exact, in [0, 2^64)
  const double whole = floor(pm);
  *out = static_cast<unsigned long long>(whole) + static_cast<unsigned long long>(llround((pm - whole) + e));
  return true;
}

}  // namespace

bool rope_turn_table(double theta, int head_dim, unsigned long long* F) {
  if (!(theta > 0.0) || !std::isfinite(theta) || (head_dim != 64 && head_dim != 128)) return false;
  for (int i = 0; i < head_dim / 2; ++i)
    if (!turn_fraction_0p64(pow(theta, -2.0 * i / head_dim), &F[i])) return false;
  return true;
}

namespace {

// The frequency table of the last (theta, head_dim) seen by this host thread (validated by
// the entry points, which refuse a theta whose table does not build).
const RopeFreqs& rope_freqs(double theta, int head_dim) {
  thread_local RopeFreqs table;
  thread_local double t_theta = -1.0;
  thread_local int t_dim = -1;
  if (theta != t_theta || head_dim != t_dim) {
    for (int i = 0; i < kMaxHeadDim / 2; ++i) table.F[i] = 0ull;
    rope_turn_table(theta, head_dim, table.F);
    t_theta = theta;
    t_dim = head_dim;
  }
  return table;
}

}  // namespace

cudaError_t launch_kv_append(const AppendArgs& a, cudaStream_t stream) {
  if (a.num_tokens == 0) return cudaSuccess;
  const RopeFreqs& fr = rope_freqs(a.theta, a.head_dim);
  constexpr int kTokensPerCta = kAppendWarps / kWarpsPerToken;
  const dim3 grid(static_cast<unsigned>((a.num_tokens + kTokensPerCta - 1) / kTokensPerCta));
  AppendSrc src;
  src.positions = a.positions;
  src.slots = a.slots;
  src.qsl = a.qsl;
  src.ctxl = a.context_lens;
  src.bt = a.block_tables;
  src.bt_stride = a.bt_stride;
  src.max_blocks = a.max_blocks;
  src.num_seqs = a.num_seqs;
  src.bs_log2 = a.bs_log2;
  src.pos_out = a.positions_out;
  src.slot_out = a.slots_out;
  record_kernel_event(PKV_KERNEL_APPEND, false, stream);
  auto* kernel = a.head_dim == 128 ? kv_append_kernel<128> : kv_append_kernel<64>;
  const cudaError_t e = launch_pdl(
      kernel, grid, dim3(kAppendWarps * 32), 0, stream,
      static_cast<bf16*>(a.q), a.q_st, a.q_sh, static_cast<const bf16*>(a.k), a.k_st, a.k_sh,
      static_cast<const bf16*>(a.v), a.v_st, a.v_sh, src, static_cast<bf16*>(a.k_cache),
      static_cast<bf16*>(a.v_cache), a.num_tokens, a.num_slots, a.hq, a.hkv, fr, a.err);
  record_kernel_event(PKV_KERNEL_APPEND, true, stream);
  return e;
}

}  // namespace pkv
