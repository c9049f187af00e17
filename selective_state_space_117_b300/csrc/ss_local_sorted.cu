// The chunked scan's local pass over channels grouped by decay speed, one warp per
// (32 channels, batch row, chunk), each state of the group dropped from the moment its
// weights underflow.
//
// The local pass only has to produce each chunk's zero-start end state
//     H[n] = sum_s exp(A[n] R_s) * w_s * B_s[n] * u_s,   R_s = sum of dt after step s in the chunk
// (w_s = dt_s for the Euler input weight; the zero-order hold replaces w_s exp(A R_s) by
// (exp(A (R_s + dt_s)) - exp(A R_s)) / A).  Walking the chunk backward from its end, R only
// grows (dt = softplus(.) >= 0), so once A[n] R log2(e) < -127 every remaining weight of state n
// is below 2^-127 and ex2.approx.ftz returns exactly 0: the remaining terms of state n add exact
// zeros.  A warp therefore skips a group of 4 states for a whole 16-step tile when that holds at
// the tile's later end for all of them in all 32 of its channels, and stops when it holds for
// every state; the sums it writes are bitwise those of the full walk.  (The chunk's dt sum it writes is then partial, but
// the carry pass only uses it through exp(A[n] * sum), which underflows to the same 0.)
//
// How much a warp can skip depends on its slowest channel, so the channels are first put in order
// of decay speed (order_channels_kernel: a counting sort of softplus(delta_bias[d]) * min_n |A[d,n]|
// into buckets a factor sqrt(2) wide, slowest first), and warp g takes the g-th 32 of that order.
// The order only changes which channels share a warp, never a channel's own arithmetic.  Slow
// groups come first in the grid, so the long items start first and the fast ones fill in behind.
//
// Data movement: a warp is its own block (no block barriers).  Each lane copies its channel's u and
// delta rows of a tile, and one 16-byte piece of the tile's B rows, with cp.async into a ring of
// kLsSlots tiles; bf16 B rows are widened once per tile into an fp32 [state][step] tile that
// every lane reads as broadcast 16-byte loads.  Per state and pair of steps: one packed multiply
// for the exponent, two MUFU.EX2, one packed multiply for the input term, one packed fma.
#include <type_traits>

#include "ss_kernels.cuh"
#include "ss_launch.h"

namespace ssk {

namespace {

#ifndef SS_LS_SLOTS
#define SS_LS_SLOTS 4
#endif
#ifndef SS_LS_MINBLOCKS
#define SS_LS_MINBLOCKS 12
#endif
constexpr int kLsSteps = 16;           // steps per tile
constexpr int kLsSlots = SS_LS_SLOTS;  // tiles in flight per warp
constexpr int kBuckets = 64;
constexpr unsigned kFull = 0xffffffffu;
constexpr float kDeadArg = -127.f;     // ex2 of anything below is under 2^-127: 0 after flushing

// Speed bucket of channel d: the slowest state's decay per step at the typical step size,
// softplus(bias) * min_n(-A[d, n]), on a log scale (2 buckets per octave, slowest first).  A
// channel with a state that does not decay (-A <= 0) goes to bucket 0.
__device__ __forceinline__ int speed_bucket(const ScanArgs& a, int64_t d) {
  const int N = (int)a.dstate;
  float rate = INFINITY;
  for (int n = 0; n < N; ++n) rate = fminf(rate, -a.A[d * N + n]);
  if (!(rate > 0.f)) return 0;
  const float key = softplus(a.delta_bias ? a.delta_bias[d] : 0.f) * rate;
  if (!(key > 0.f)) return 0;
  const int b = (int)floorf(__log2f(key) * 2.f) + 48;
  return min(max(b, 1), kBuckets - 1);
}

// perm[0 .. dim) = the channels in increasing speed bucket (one block).
__global__ void __launch_bounds__(1024) order_channels_kernel(const ScanArgs a, int* perm) {
  __shared__ int cnt[kBuckets];
  const int tid = threadIdx.x;
  if (tid < kBuckets) cnt[tid] = 0;
  __syncthreads();
  for (int64_t d = tid; d < a.dim; d += blockDim.x) atomicAdd(&cnt[speed_bucket(a, d)], 1);
  __syncthreads();
  if (tid == 0) {
    int run = 0;
    for (int b = 0; b < kBuckets; ++b) {
      const int c = cnt[b];
      cnt[b] = run;
      run += c;
    }
  }
  __syncthreads();
  for (int64_t d = tid; d < a.dim; d += blockDim.x) perm[atomicAdd(&cnt[speed_bucket(a, d)], 1)] = (int)d;
}

template <int NT, bool BF>
struct LsLayout {
  static constexpr int ES = In<BF>::kBytes;
  static constexpr int RB = kLsSteps * ES;     // bytes of one row of a tile: 32 (bf16) or 64 (fp32)
  static constexpr int CH = RB / 16;           // 16-byte pieces per row
  static constexpr int kIn = 32 * RB;          // u or delta rows of the warp's 32 channels, piece-major
  static constexpr int kB = NT * RB;           // the tile's raw B rows, [state][step]
  static constexpr int kSlot = 2 * kIn + kB;
  static constexpr int kBf = BF ? NT * kLsSteps * 4 : 0;   // B widened to fp32 (bf16 inputs)
  static constexpr int kBytes = kLsSlots * kSlot + kBf;
  static constexpr int kBPieces = NT * CH;     // 16-byte pieces of raw B per tile
};

// A lane's row of a tile (16 steps) as 8 pairs of steps: its 16-byte pieces are stored
// piece-major ([piece][lane]), so the 32 lanes' reads of one piece are 512 contiguous bytes.
template <bool BF>
__device__ __forceinline__ void row_pairs(const unsigned char* arr, int lane, f2 (&v)[kLsSteps / 2]) {
  if constexpr (BF) {
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const uint4 r = *reinterpret_cast<const uint4*>(arr + c * 512 + lane * 16);
      v[4 * c] = bf16x2(r.x);
      v[4 * c + 1] = bf16x2(r.y);
      v[4 * c + 2] = bf16x2(r.z);
      v[4 * c + 3] = bf16x2(r.w);
    }
  } else {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const float4 r = *reinterpret_cast<const float4*>(arr + c * 512 + lane * 16);
      v[2 * c] = pk(r.x, r.y);
      v[2 * c + 1] = pk(r.z, r.w);
    }
  }
}

// States are taken in groups of kLsGroup: a group is skipped for a tile only when all of its
// states are dead in every channel of the warp (a dead state inside a live group adds exact
// zeros).  One vote per group, and the group's states are independent chains that the
// compiler interleaves.
constexpr int kLsGroup = 4;

template <int NT, bool BF, bool ZOH>
__global__ void __launch_bounds__(32, SS_LS_MINBLOCKS) local_sorted_kernel(const ScanArgs a, const int* __restrict__ perm,
                                                          int64_t kchunks) {
  using L = In<BF>;
  using Lay = LsLayout<NT, BF>;
  constexpr int S = kLsSlots;
  constexpr int NPAIR = kLsSteps / 2;
  __shared__ __align__(128) unsigned char sm[Lay::kBytes];

  const int lane = threadIdx.x;
  const int64_t items_per_group = a.batch * kchunks;
  const int64_t g = blockIdx.x / items_per_group, rem = blockIdx.x % items_per_group;
  const int64_t b = rem / kchunks, k = rem % kchunks;
  const int N = (int)a.dstate;
  const int64_t slot = g * 32 + lane;
  const bool active = slot < a.dim;
  const int64_t d = perm[active ? slot : a.dim - 1];
  const int64_t bd = b * a.dim + d;
  const int64_t t_begin = k * a.chunk_len;
  const int ntiles = (int)(a.chunk_len / kLsSteps);   // the launcher guarantees whole tiles

  // Per-state constants: A' = A * log2(e) (0 for padding states, which are never processed),
  // and each group's slowest A' (the last of its states to die).
  constexpr int NG = (NT + kLsGroup - 1) / kLsGroup;
  float Ap[NT], iAs[NT], gmax[NG];
  float amax = -INFINITY;
#pragma unroll
  for (int gi = 0; gi < NG; ++gi) gmax[gi] = -INFINITY;
#pragma unroll
  for (int n = 0; n < NT; ++n) {
    const float an = (n < N) ? a.A[d * N + n] : 0.f;
    Ap[n] = an * kLog2e;
    iAs[n] = an != 0.f ? 1.f / an : 0.f;
    if (n < N) {
      amax = fmaxf(amax, Ap[n]);
      gmax[n / kLsGroup] = fmaxf(gmax[n / kLsGroup], Ap[n]);
    }
  }
  const float bias = a.delta_bias ? a.delta_bias[d] : 0.f;
  const f2 bias2 = pk(bias, bias);
  const bool may_stop = a.softplus != 0;

  // Copies of time tile (ntiles - 1 - i) into ring slot i % S (the walk goes backward).
  const char* urow = static_cast<const char*>(a.u) + (bd * a.seqlen + t_begin) * Lay::ES;
  const char* drow = static_cast<const char*>(a.delta) + (bd * a.seqlen + t_begin) * Lay::ES;
  const char* bbase = static_cast<const char*>(a.B) + (b * N * a.seqlen + t_begin) * Lay::ES;
  auto issue = [&](int i) {
    unsigned char* s = sm + (i % S) * Lay::kSlot;
    const int64_t off = (int64_t)(ntiles - 1 - i) * Lay::RB;
#pragma unroll
    for (int c = 0; c < Lay::CH; ++c) {
      cp_async16(smem_addr(s + c * 512 + lane * 16), urow + off + c * 16);
      cp_async16(smem_addr(s + Lay::kIn + c * 512 + lane * 16), drow + off + c * 16);
    }
#pragma unroll
    for (int q0 = 0; q0 < Lay::kBPieces; q0 += 32) {
      const int q = q0 + lane, n = q / Lay::CH, c = q % Lay::CH;
      if (q < Lay::kBPieces && n < N)
        cp_async16(smem_addr(s + 2 * Lay::kIn + q * 16), bbase + (int64_t)n * a.seqlen * Lay::ES + off + c * 16);
    }
  };
  // Raw B rows of padding states stay zero in every slot.
#pragma unroll
  for (int q0 = 0; q0 < Lay::kBPieces; q0 += 32) {
    const int q = q0 + lane;
    if (q < Lay::kBPieces && q / Lay::CH >= N)
      for (int s = 0; s < S; ++s)
        *reinterpret_cast<uint4*>(sm + s * Lay::kSlot + 2 * Lay::kIn + q * 16) = make_uint4(0, 0, 0, 0);
  }
#pragma unroll
  for (int i = 0; i < S - 1; ++i) {
    if (i < ntiles) issue(i);
    cp_async_commit();
  }

  f2 acc[NT];
#pragma unroll
  for (int n = 0; n < NT; ++n) acc[n] = pk(0.f, 0.f);
  float R = 0.f;   // sum of dt after the current tile

  for (int i = 0; i < ntiles; ++i) {
    // Every state of every channel of the warp has underflowed: the rest of the chunk adds zeros.
    if (may_stop && !__any_sync(kFull, active && amax * R >= kDeadArg)) break;
    if (i + S - 1 < ntiles) issue(i + S - 1);
    cp_async_commit();
    cp_async_wait<S - 1>();
    __syncwarp();
    const unsigned char* s = sm + (i % S) * Lay::kSlot;
    const float* Bt;
    if constexpr (BF) {
      // Widen the tile's B rows to fp32: lane q converts piece q (state q / 2, steps 8 (q % 2) ..).
      float* bf = reinterpret_cast<float*>(sm + S * Lay::kSlot);
#pragma unroll
      for (int q0 = 0; q0 < Lay::kBPieces; q0 += 32) {
        const int q = q0 + lane;
        if (q < Lay::kBPieces) {
          const uint4 r = *reinterpret_cast<const uint4*>(s + 2 * Lay::kIn + q * 16);
          float4* o = reinterpret_cast<float4*>(bf + q * 8);
          o[0] = make_float4(bf16_lo(r.x), bf16_hi(r.x), bf16_lo(r.y), bf16_hi(r.y));
          o[1] = make_float4(bf16_lo(r.z), bf16_hi(r.z), bf16_lo(r.w), bf16_hi(r.w));
        }
      }
      __syncwarp();
      Bt = bf;
    } else {
      Bt = reinterpret_cast<const float*>(s + 2 * Lay::kIn);
    }

    // The tile's step scalars as pairs of steps (2p, 2p + 1): dt, dt * u (or u for the hold), and
    // R_s, the sum of dt after step s (from the chunk's end), built from the tile's end backward.
    f2 dt2[NPAIR], w2[NPAIR], R2[NPAIR];
    {
      f2 xr[NPAIR], ur[NPAIR];
      row_pairs<BF>(s + Lay::kIn, lane, xr);
      row_pairs<BF>(s, lane, ur);
#pragma unroll
      for (int p = 0; p < NPAIR; ++p) {
        const f2 x = add2(xr[p], bias2);
        dt2[p] = a.softplus ? softplus2(x) : x;
        w2[p] = ZOH ? ur[p] : mul2(dt2[p], ur[p]);
      }
    }
    // Suffix sums over the tile's 8 pairs as a 3-level tree (instead of a chain of 16 adds):
    // after[p] = sum of dt over pairs p+1 .. 7.
    const float R_in = R;
    {
      float ps[NPAIR], after[NPAIR];
#pragma unroll
      for (int p = 0; p < NPAIR; ++p) ps[p] = lo(dt2[p]) + hi(dt2[p]);
      const float s67 = ps[6] + ps[7], s45 = ps[4] + ps[5], s23 = ps[2] + ps[3], s4567 = s45 + s67;
      after[7] = 0.f;
      after[6] = ps[7];
      after[5] = s67;
      after[4] = ps[5] + s67;
      after[3] = s4567;
      after[2] = ps[3] + s4567;
      after[1] = s23 + s4567;
      after[0] = (ps[1] + s23) + s4567;
#pragma unroll
      for (int p = 0; p < NPAIR; ++p) {
        const float r_hi = R_in + after[p];
        R2[p] = pk(r_hi + hi(dt2[p]), r_hi);
      }
      R = R_in + (ps[0] + after[0]);
    }

#pragma unroll
    for (int gi = 0; gi < NG; ++gi) {
      if (gi * kLsGroup >= N) break;
      if (may_stop && !__any_sync(kFull, active && gmax[gi] * R_in >= kDeadArg)) continue;
#pragma unroll
      for (int n = gi * kLsGroup; n < (gi + 1) * kLsGroup && n < NT; ++n) {
        if (n >= N) break;
        const float4* brow = reinterpret_cast<const float4*>(Bt + n * kLsSteps);
        const f2 A2 = pk(Ap[n], Ap[n]);
        f2 sum = acc[n];
        if constexpr (ZOH) {
          // Weights at the 17 points R_{-1} = R (before the tile), R_0, ..., R_15: the hold weight
          // of step s is (w(R_{s-1}) - w(R_s)) / A with w(R) = exp(A R).
          const f2 iA2 = pk(iAs[n], iAs[n]);
          float w_prev = ex2(Ap[n] * R);   // w(R_{-1})
#pragma unroll
          for (int p = 0; p < NPAIR; ++p) {
            const float4 bv = brow[p >> 1];
            const f2 Bp = (p & 1) ? pk(bv.z, bv.w) : pk(bv.x, bv.y);
            const f2 wc = ex2x2(mul2(R2[p], A2));
            const f2 wn = pk(w_prev, lo(wc));
            w_prev = hi(wc);
            const f2 hold = hold_between2(wn, wc, mul2(dt2[p], A2), dt2[p], iA2);
            sum = fma2(hold, mul2(w2[p], Bp), sum);
          }
        } else {
#pragma unroll
          for (int p = 0; p < NPAIR; ++p) {
            const float4 bv = brow[p >> 1];
            const f2 Bp = (p & 1) ? pk(bv.z, bv.w) : pk(bv.x, bv.y);
            sum = fma2(ex2x2(mul2(R2[p], A2)), mul2(w2[p], Bp), sum);
          }
        }
        acc[n] = sum;
      }
    }
    __syncwarp();   // every lane is done with this slot and the fp32 B tile before they are refilled
  }
  cp_async_wait<0>();   // no copy may still be landing in shared memory when the warp exits

  if (!active) return;
  const int64_t BD = a.batch * a.dim;
  a.ws_S[k * BD + bd] = R;
  float* H = a.ws_H + (k * BD + bd) * N;
#pragma unroll
  for (int n = 0; n < NT; ++n)
    if (n < N) H[n] = lo(acc[n]) + hi(acc[n]);
}

template <int NT, bool BF, bool ZOH>
int go_local_sorted(const ScanArgs& a, int64_t kchunks, cudaStream_t s) {
  const int64_t groups = (a.dim + 31) / 32;
  const int64_t items = groups * a.batch * kchunks;
  order_channels_kernel<<<1, 1024, 0, s>>>(a, a.perm);
  local_sorted_kernel<NT, BF, ZOH><<<(unsigned)items, 32, 0, s>>>(a, a.perm, kchunks);
  return 0;
}

}  // namespace

bool local_sorted_available(const ScanArgs& a, bool bf16) {
  (void)bf16;
  const int64_t kchunks = a.local_chunks;
  if (kchunks < 1 || !a.perm) return false;
  if (a.dstate < 1 || a.dstate > 16 || !a.vec || !a.vec_bc || a.chunk_len % kLsSteps != 0) return false;
  if (a.dim > (int64_t)INT32_MAX) return false;
  const int64_t items = (a.dim + 31) / 32 * a.batch * kchunks;
  return items <= (int64_t)INT32_MAX;
}

int launch_local_sorted(const ScanArgs& a, bool bf16, cudaStream_t s) {
  const int64_t kchunks = a.local_chunks;
  const int N = (int)a.dstate;
  auto go = [&](auto nt) -> int {
    constexpr int NT = decltype(nt)::value;
    if (bf16) return a.zoh ? go_local_sorted<NT, true, true>(a, kchunks, s) : go_local_sorted<NT, true, false>(a, kchunks, s);
    return a.zoh ? go_local_sorted<NT, false, true>(a, kchunks, s) : go_local_sorted<NT, false, false>(a, kchunks, s);
  };
  if (N <= 4) return go(std::integral_constant<int, 4>{});
  if (N <= 8) return go(std::integral_constant<int, 8>{});
  return go(std::integral_constant<int, 16>{});
}

}  // namespace ssk
