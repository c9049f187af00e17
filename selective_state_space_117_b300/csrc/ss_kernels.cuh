// Selective scan kernels over (batch row, channel, chunk) units (sm_103a).
//
// Work decomposition: one thread owns one (batch row b, channel d, chunk k)
// and keeps that channel's N states in registers for the whole chunk, so the
// (batch, L, dim, N) expanded state never leaves the SM ("Kernel fusion",
// "Mamba: Linear-Time Sequence Modeling with Selective State Spaces").  A
// block is kCh consecutive channels of one (b, k).  All of them read the same
// B_t and C_t, which the block stages through shared memory as fp32 tiles of
// Tile<NT>::kSteps steps (double-buffered; the next tile's raw values are
// fetched into registers while the current tile is consumed) and every thread
// reads as broadcast 16-byte loads.  u, delta and z are read along each
// thread's own row as 16-byte vectors, one group of 8 steps ahead of use; y is
// written the same way.
//
// Arithmetic runs on state pairs with the packed f32x2 instructions: per pair
// and step one mul (dt*A'), two MUFU.EX2, one mul (du*B), one fma (the state)
// and one fma (the readout C*h), where A' = A*log2(e).
//
// scan_kernel modes:
//   kFull   start from h = 0 (or h0), write y and (optionally) the final state
//   kFixup  start from the carried-in state in the workspace, write y, and the final
//           state from the last chunk
// local_kernel is the first phase of the chunked scan (see its comment).
#pragma once

#include "ss_device.cuh"
#include "ss_types.h"

namespace ssk {

// B/C tile geometry: kSteps * NT = 512 values per array, so one tile is one
// 8-step segment of B and one of C per thread (kCh = 64 threads).
template <int NT>
struct Tile {
  static constexpr int kSteps = 512 / NT;
  static constexpr int kSegs = kSteps / kGroup;  // 8-step segments per state row
  static_assert(NT * kSegs == kCh, "one B segment and one C segment per thread");
};

// Shared-memory ring of 8-step input groups: slots, and how many groups ahead they are filled.
constexpr int kStages = 4;
constexpr int kAhead = kStages - 1;

// Register ceiling: the state count decides how many blocks of kCh threads
// must fit on an SM.  NT <= 16: 6 blocks (12 warps, 3 per scheduler) leave
// 168 registers per thread, which measured faster than 8 blocks at 128
// registers (the compiler keeps more of each 8-step group in flight); the
// launcher may run fewer blocks per SM to even out the last wave
// (ss_occupancy.cuh).
template <int NT, bool BF>
struct MinBlocks {
  static constexpr int value = NT <= 16 ? 6 : (NT == 32 ? 5 : 3);
};

// One 8-step segment of a B or C state row, fetched raw into registers and
// stored transposed ([t][n], fp32) into a shared-memory tile.
template <int NT, bool BF>
struct Segment {
  using L = In<BF>;
  typename L::Raw8 raw;

  // Row n of `src` (offset `row0` = (b, n, 0)), steps [t, t + 8) clipped to t_end.
  __device__ __forceinline__ void load(const void* src, int64_t off, bool ok_row, int64_t t, int64_t t_end, bool vec) {
    if (ok_row && vec && t + kGroup <= t_end) {
      raw = L::load8(src, off);
    } else {
      float v[kGroup];
#pragma unroll
      for (int j = 0; j < kGroup; ++j) v[j] = (ok_row && t + j < t_end) ? L::one(src, off + j) : 0.f;
      raw = L::pack8(v);
    }
  }
  __device__ __forceinline__ void store(float* tile, int n, int tseg) const {
#pragma unroll
    for (int p = 0; p < kGroup / 2; ++p) {
      const f2 v = L::pair(raw, p);
      tile[(tseg * kGroup + 2 * p) * NT + n] = lo(v);
      tile[(tseg * kGroup + 2 * p + 1) * NT + n] = hi(v);
    }
  }
};

// The unit of work of this block: rows, time range and channel.
struct Unit {
  int64_t b, d, k, bd, row, bc_row, t_begin, t_end;
  bool active;
};

__device__ __forceinline__ Unit unit_of(const ScanArgs& a) {
  Unit w;
  const int ct = blockIdx.x % a.ctiles;
  w.k = blockIdx.x / a.ctiles;
  w.b = blockIdx.y;
  w.d = (int64_t)ct * kCh + threadIdx.x;
  w.active = w.d < a.dim;
  w.t_begin = w.k * a.chunk_len;
  w.t_end = min(a.seqlen, w.t_begin + a.chunk_len);
  w.bd = w.b * a.dim + (w.active ? w.d : 0);
  w.row = w.bd * a.seqlen;
  w.bc_row = w.b * a.dstate * a.seqlen;
  return w;
}

// Debug-build bounds of a unit: its rows of u/delta/z/y, of B/C, its A row, its state rows
// (h0, last_state) and its workspace entries.  Always true in the normal build.
__device__ __forceinline__ bool unit_ok(const ScanArgs& a, const Unit& w) {
  const int64_t N = a.dstate, BD = a.batch * a.dim;
  bool ok = span_ok(a.err, w.row + w.t_begin, w.t_end - w.t_begin, BD * a.seqlen);
  ok = span_ok(a.err, w.bc_row, N * a.seqlen, a.batch * N * a.seqlen) && ok;
  ok = span_ok(a.err, w.d * N, N, a.dim * N) && ok;
  ok = span_ok(a.err, w.bd * N, N, BD * N) && ok;
  if (a.ws_H) ok = span_ok(a.err, (w.k * BD + w.bd) * N, N, a.nchunks * BD * N) && ok;
  if (a.ws_S) ok = span_ok(a.err, w.k * BD + w.bd, 1, a.nchunks * BD) && ok;
  return ok;
}

// Per-step scalars of one 8-step group: dt, du = dt*u as pairs (steps 2p, 2p+1).
template <bool BF>
__device__ __forceinline__ void step_scalars(const typename In<BF>::Raw8& ru, const typename In<BF>::Raw8& rd,
                                             f2 bias2, int softplus, f2 (&dt2)[4], f2 (&du2)[4]) {
  using L = In<BF>;
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    const f2 x = add2(L::pair(rd, p), bias2);
    dt2[p] = softplus ? softplus2(x) : x;
    du2[p] = mul2(dt2[p], L::pair(ru, p));
  }
}

// One full 8-step group of the forward recurrence for this thread's channel:
// inputs as raw 8-element rows (u, delta, z), B and C of the 8 steps as fp32
// rows of NT values at cB and cC, the state h updated in place, and the 8
// outputs (skip term and gate applied) returned as pairs in y2.
// One state pair's update h = Abar h + (input weight) B u for one step:
// Euler weight dt (du = dt u), or the zero-order-hold weight (hold2).
template <bool ZOH>
__device__ __forceinline__ f2 step_pair(f2 h, f2 A2, f2 iA2, f2 dtp, f2 dup, f2 upp, f2 Bp) {
  const f2 arg = mul2(dtp, A2);
  const f2 e = ex2x2(arg);
  if constexpr (ZOH) return fma2(e, h, mul2(hold2(arg, e, dtp, iA2), mul2(upp, Bp)));
  return fma2(e, h, mul2(dup, Bp));
}

// The readout sum over state pairs runs as one chain of fused multiply-adds, or with
// TWO_CHAINS as two (even and odd pairs) added at the end: one more instruction per
// step, half the chain's latency.  Two chains pay where few warps share an SM (the
// full-sequence scan of a layer with few channels per SM), one where many do (the
// chunked fix-up pass).
template <int NT, bool BF, bool HAS_Z, bool ZOH, bool TWO_CHAINS = false>
__device__ __forceinline__ void scan_group(const typename In<BF>::Raw8& cu, const typename In<BF>::Raw8& rd,
                                           const typename In<BF>::Raw8& cz, f2 bias2, f2 D2, int softplus,
                                           const f2 (&A2)[NT / 2], const f2 (&iA2)[NT / 2], f2 (&h)[NT / 2],
                                           const float* cB, const float* cC, f2 (&y2)[4]) {
  using L = In<BF>;
  constexpr int NP = NT / 2;
  f2 dt2[4], du2[4];
  step_scalars<BF>(cu, rd, bias2, softplus, dt2, du2);
  float yo[kGroup];
#pragma unroll
  for (int j = 0; j < kGroup; ++j) {
    const float dt = (j & 1) ? hi(dt2[j >> 1]) : lo(dt2[j >> 1]);
    const float du = (j & 1) ? hi(du2[j >> 1]) : lo(du2[j >> 1]);
    f2 upp = pk(0.f, 0.f);
    if (ZOH) {
      const f2 u2 = L::pair(cu, j >> 1);
      const float uu = (j & 1) ? hi(u2) : lo(u2);
      upp = pk(uu, uu);
    }
    const f2 dtp = pk(dt, dt), dup = pk(du, du);
    const float* rb = cB + j * NT;
    const float* rc = cC + j * NT;
    f2 acc, acc1;
#pragma unroll
    for (int q = 0; q < NP; q += 2) {
      const float4 bv = *reinterpret_cast<const float4*>(rb + 2 * q);
      const float4 cv = *reinterpret_cast<const float4*>(rc + 2 * q);
      h[q] = step_pair<ZOH>(h[q], A2[q], iA2[q], dtp, dup, upp, pk(bv.x, bv.y));
      acc = q == 0 ? mul2(pk(cv.x, cv.y), h[q]) : fma2(pk(cv.x, cv.y), h[q], acc);
      h[q + 1] = step_pair<ZOH>(h[q + 1], A2[q + 1], iA2[q + 1], dtp, dup, upp, pk(bv.z, bv.w));
      if constexpr (TWO_CHAINS) acc1 = q == 0 ? mul2(pk(cv.z, cv.w), h[q + 1]) : fma2(pk(cv.z, cv.w), h[q + 1], acc1);
      else acc = fma2(pk(cv.z, cv.w), h[q + 1], acc);
    }
    if constexpr (TWO_CHAINS) acc = add2(acc, acc1);
    yo[j] = lo(acc) + hi(acc);
  }
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    y2[p] = fma2(D2, L::pair(cu, p), pk(yo[2 * p], yo[2 * p + 1]));
    if (HAS_Z) y2[p] = mul2(y2[p], silu2(L::pair(cz, p)));
  }
}

template <int NT, bool BF, bool HAS_Z, int MODE, bool ZOH>
__global__ void __launch_bounds__(kCh, (MinBlocks<NT, BF>::value)) scan_kernel(const ScanArgs a) {
  using L = In<BF>;
  using T = Tile<NT>;
  constexpr int NP = NT / 2;
  constexpr int NA = HAS_Z ? 3 : 2;             // input arrays in the ring: u, delta (, z)
  using RingT = Ring<BF, NA, kCh, kStages>;
  __shared__ __align__(16) float sB[2][T::kSteps * NT];
  __shared__ __align__(16) float sC[2][T::kSteps * NT];
  __shared__ __align__(16) unsigned char sIn[RingT::kBytes];

  const int tid = threadIdx.x;
  Unit w = unit_of(a);
  w.active = w.active && unit_ok(a, w);
  const int N = (int)a.dstate;

  // Padding states n >= N keep B = C = 0 (their staged values are zero), A = 0 and h = 0.
  f2 A2[NP], iA2[NP], h[NP];
  const float* Arow = a.A + (w.active ? w.d : 0) * N;
#pragma unroll
  for (int q = 0; q < NP; ++q) {
    const int n0 = 2 * q, n1 = 2 * q + 1;
    const float a0 = (w.active && n0 < N) ? Arow[n0] : 0.f, a1 = (w.active && n1 < N) ? Arow[n1] : 0.f;
    A2[q] = pk(a0 * kLog2e, a1 * kLog2e);
    iA2[q] = pk(a0 != 0.f ? 1.f / a0 : 0.f, a1 != 0.f ? 1.f / a1 : 0.f);
    float h0 = 0.f, h1 = 0.f;
    const float* H = nullptr;
    if (MODE == kFixup) H = a.ws_H + (w.k * a.batch * a.dim + w.bd) * N;  // carry-in of this chunk
    else if (a.h0) H = a.h0 + w.bd * N;                             // caller's initial state
    if (H && w.active) {
      if (n0 < N) h0 = H[n0];
      if (n1 < N) h1 = H[n1];
    }
    h[q] = pk(h0, h1);
  }
  const float bias = (a.delta_bias && w.active) ? a.delta_bias[w.d] : 0.f;
  const float Dd = (a.D && w.active) ? a.D[w.d] : 0.f;
  const f2 bias2 = pk(bias, bias), D2 = pk(Dd, Dd);

  // This thread's B and C segment of every tile.
  const int sn = tid % NT, tseg = tid / NT;
  const bool srow = sn < N;
  const int64_t soff = w.bc_row + (int64_t)sn * a.seqlen + tseg * kGroup;
  Segment<NT, BF> segB, segC;
  segB.load(a.B, soff + w.t_begin, srow, w.t_begin + tseg * kGroup, w.t_end, a.vec_bc);
  segC.load(a.C, soff + w.t_begin, srow, w.t_begin + tseg * kGroup, w.t_end, a.vec_bc);
  segB.store(sB[0], sn, tseg);
  segC.store(sC[0], sn, tseg);

  // Full 8-step groups go through the ring (vector path); the rest is scalar.
  const int nfull = (w.active && a.vec) ? (int)((w.t_end - w.t_begin) / kGroup) : 0;
  RingT ring;
  ring.base = smem_addr(sIn) + tid * 16;
  ring.src[0] = static_cast<const char*>(L::addr(a.u, w.row + w.t_begin));
  ring.src[1] = static_cast<const char*>(L::addr(a.delta, w.row + w.t_begin));
  if (HAS_Z) ring.src[NA - 1] = static_cast<const char*>(L::addr(a.z, w.row + w.t_begin));
  ring.step = kGroup * L::kBytes;
  if (nfull > 0)
    for (int gi = 0; gi < kAhead; ++gi) {
      if (gi < nfull) ring.put(gi);
      cp_async_commit();
    }
  __syncthreads();

  int buf = 0;
  for (int64_t tt0 = w.t_begin; tt0 < w.t_end; tt0 += T::kSteps) {
    const int tn = (int)min((int64_t)T::kSteps, w.t_end - tt0);
    const int64_t nx0 = tt0 + T::kSteps;
    const bool more = nx0 < w.t_end;
    if (more) {
      segB.load(a.B, soff + nx0, srow, nx0 + tseg * kGroup, w.t_end, a.vec_bc);
      segC.load(a.C, soff + nx0, srow, nx0 + tseg * kGroup, w.t_end, a.vec_bc);
    }
    if (w.active) {
      const float* cB = sB[buf];
      const float* cC = sC[buf];
      for (int g = 0; g < tn; g += kGroup) {
        const int64_t t = tt0 + g;
        const int gi = (int)((t - w.t_begin) / kGroup);
        if (gi < nfull) {
          if (gi + kAhead < nfull) ring.put(gi + kAhead);
          cp_async_commit();
          cp_async_wait<kAhead>();
          const typename L::Raw8 cu = ring.get(gi, 0);
          const typename L::Raw8 rd = ring.get(gi, 1);
          typename L::Raw8 cz{};
          if (HAS_Z) cz = ring.get(gi, NA - 1);
          f2 y2[4];
          scan_group<NT, BF, HAS_Z, ZOH, MODE == kFull>(cu, rd, cz, bias2, D2, a.softplus, A2, iA2, h, cB + g * NT,
                                                        cC + g * NT, y2);
          float4* qy = reinterpret_cast<float4*>(a.y + w.row + t);
          qy[0] = make_float4(lo(y2[0]), hi(y2[0]), lo(y2[1]), hi(y2[1]));
          qy[1] = make_float4(lo(y2[2]), hi(y2[2]), lo(y2[3]), hi(y2[3]));
        } else {
          // ---- scalar path: unaligned rows or the ragged end of the sequence
          const int nv = min(kGroup, tn - g);
          for (int j = 0; j < nv; ++j) {
            const int64_t ix = w.row + t + j;
            const float uu = L::one(a.u, ix);
            const float x = L::one(a.delta, ix) + bias;
            const float dt = a.softplus ? softplus(x) : x;
            const f2 dtp = pk(dt, dt), dup = pk(dt * uu, dt * uu), upp = pk(uu, uu);
            const float* rb = cB + (g + j) * NT;
            const float* rc = cC + (g + j) * NT;
            f2 acc = pk(0.f, 0.f);
#pragma unroll
            for (int q = 0; q < NP; ++q) {
              const f2 bq = *reinterpret_cast<const f2*>(rb + 2 * q);
              const f2 cq = *reinterpret_cast<const f2*>(rc + 2 * q);
              h[q] = step_pair<ZOH>(h[q], A2[q], iA2[q], dtp, dup, upp, bq);
              acc = fma2(cq, h[q], acc);
            }
            float yv = fmaf(Dd, uu, lo(acc) + hi(acc));
            if (HAS_Z) yv *= silu(L::one(a.z, ix));
            a.y[ix] = yv;
          }
        }
      }
    }
    if (more) {
      segB.store(sB[buf ^ 1], sn, tseg);
      segC.store(sC[buf ^ 1], sn, tseg);
      __syncthreads();
      buf ^= 1;
    }
  }

  cp_async_wait<0>();
  // The final state: after the whole sequence, or after the last chunk of the chunked scan.
  if ((MODE == kFull || w.k == a.nchunks - 1) && w.active && a.last_state) {
    float* out = a.last_state + w.bd * N;
#pragma unroll
    for (int q = 0; q < NP; ++q) {
      if (2 * q < N) out[2 * q] = lo(h[q]);
      if (2 * q + 1 < N) out[2 * q + 1] = hi(h[q]);
    }
  }
}

// One state pair's term of the backward local pass at one step, with R the sum
// of dt after the step: Euler adds exp(A R) dt B u; the zero-order hold adds
// (exp(A (R + dt)) - exp(A R)) / A * B u, the first exponential being the one the
// next (earlier) step needs, so wc carries it and the hold costs no extra exp.
template <bool ZOH>
__device__ __forceinline__ void local_pair(f2& acc, f2& wc, f2 A2, f2 iA2, float R, float dt, float du, float uu,
                                           f2 Bp) {
  if constexpr (ZOH) {
    const f2 dtp = pk(dt, dt), Rn = pk(R + dt, R + dt);
    const f2 wn = ex2x2(mul2(Rn, A2));
    acc = fma2(hold_between2(wn, wc, mul2(dtp, A2), dtp, iA2), mul2(pk(uu, uu), Bp), acc);
    wc = wn;
  } else {
    acc = fma2(ex2x2(mul2(pk(R, R), A2)), mul2(pk(du, du), Bp), acc);
  }
}

// First phase of the chunked scan: for every chunk, its zero-start end state
//   Hend[n] = sum_s exp(A[n] * R_s) * dt_s * B_s[n] * u_s,   R_s = sum_{r > s in chunk} dt_r
// and the chunk's sum of dt, computed backward from the chunk's end.  With
// dt >= 0 (softplus on) R only grows, so once A[n] * R * log2(e) < -127 every
// remaining weight exp2(.) of state n is below 2^-127 and flushes to zero in
// fp32; the block stops at the first tile where that holds for every state
// of every channel.  The sum written is then partial, but every
// exp(A[n] * sum) that the carry pass forms from it underflows to zero
// exactly as the full sum's would.
template <int NT, bool BF, bool ZOH>
__global__ void __launch_bounds__(kCh, (MinBlocks<NT, BF>::value)) local_kernel(const ScanArgs a) {
  using L = In<BF>;
  using T = Tile<NT>;
  constexpr int NP = NT / 2;
  constexpr float kDead = -127.f;
  using RingT = Ring<BF, 2, kCh, kStages>;     // u, delta
  __shared__ __align__(16) float sB[2][T::kSteps * NT];
  __shared__ __align__(16) unsigned char sIn[RingT::kBytes];

  const int tid = threadIdx.x;
  Unit w = unit_of(a);
  w.active = w.active && unit_ok(a, w);
  const int N = (int)a.dstate;

  f2 A2[NP], iA2[NP], wc[NP], acc[NP];
  float amax = -1e30f;  // the slowest decay of this channel (padding states never count)
  const float* Arow = a.A + (w.active ? w.d : 0) * N;
#pragma unroll
  for (int q = 0; q < NP; ++q) {
    const int n0 = 2 * q, n1 = 2 * q + 1;
    const float an0 = (w.active && n0 < N) ? Arow[n0] : 0.f, an1 = (w.active && n1 < N) ? Arow[n1] : 0.f;
    const float a0 = an0 * kLog2e, a1 = an1 * kLog2e;
    A2[q] = pk(a0, a1);
    iA2[q] = pk(an0 != 0.f ? 1.f / an0 : 0.f, an1 != 0.f ? 1.f / an1 : 0.f);
    wc[q] = pk(1.f, 1.f);  // exp(A R) at R = 0 (zero-order hold only)
    if (n0 < N) amax = fmaxf(amax, a0);
    if (n1 < N) amax = fmaxf(amax, a1);
    acc[q] = pk(0.f, 0.f);
  }
  const float bias = (a.delta_bias && w.active) ? a.delta_bias[w.d] : 0.f;
  const f2 bias2 = pk(bias, bias);
  const bool may_stop = a.softplus != 0;
  float R = 0.f;

  const int sn = tid % NT, tseg = tid / NT;
  const bool srow = sn < N;
  const int64_t soff = w.bc_row + (int64_t)sn * a.seqlen + tseg * kGroup;
  const int64_t ntiles = (w.t_end - w.t_begin + T::kSteps - 1) / T::kSteps;
  Segment<NT, BF> segB;

  int64_t tt0 = w.t_begin + (ntiles - 1) * T::kSteps;
  segB.load(a.B, soff + tt0, srow, tt0 + tseg * kGroup, w.t_end, a.vec_bc);
  segB.store(sB[0], sn, tseg);
  __syncthreads();

  // Groups are taken from the chunk's end backward; with aligned rows and a
  // chunk of whole groups every group goes through the ring, else none does.
  const int ngr = (int)((w.t_end - w.t_begin + kGroup - 1) / kGroup);
  const bool ring_on = w.active && a.vec && (w.t_end - w.t_begin) % kGroup == 0;
  RingT ring;  // group j of the ring is the j-th group from the chunk's end
  ring.base = smem_addr(sIn) + tid * 16;
  ring.src[0] = static_cast<const char*>(L::addr(a.u, w.row + w.t_end - kGroup));
  ring.src[1] = static_cast<const char*>(L::addr(a.delta, w.row + w.t_end - kGroup));
  ring.step = -(int64_t)(kGroup * L::kBytes);
  if (ring_on)
    for (int j = 0; j < kAhead; ++j) {
      if (j < ngr) ring.put(j);
      cp_async_commit();
    }

  int buf = 0;
  for (int64_t it = ntiles - 1; it >= 0; --it, tt0 -= T::kSteps) {
    const int tn = (int)min((int64_t)T::kSteps, w.t_end - tt0);
    const bool more = it > 0;
    if (more) segB.load(a.B, soff + tt0 - T::kSteps, srow, tt0 - T::kSteps + tseg * kGroup, w.t_end, a.vec_bc);
    if (w.active) {
      const float* cB = sB[buf];
      const int ng = (tn + kGroup - 1) / kGroup;
      for (int gi = ng - 1; gi >= 0; --gi) {
        const int g = gi * kGroup;
        const int64_t t = tt0 + g;
        if (ring_on) {
          const int j = ngr - 1 - (int)((t - w.t_begin) / kGroup);
          if (j + kAhead < ngr) ring.put(j + kAhead);
          cp_async_commit();
          cp_async_wait<kAhead>();
          const typename L::Raw8 ru = ring.get(j, 0);
          const typename L::Raw8 rd = ring.get(j, 1);
          f2 dt2[4], du2[4];
          step_scalars<BF>(ru, rd, bias2, a.softplus, dt2, du2);
#pragma unroll
          for (int j = kGroup - 1; j >= 0; --j) {
            const float dt = (j & 1) ? hi(dt2[j >> 1]) : lo(dt2[j >> 1]);
            const float du = (j & 1) ? hi(du2[j >> 1]) : lo(du2[j >> 1]);
            const float uu = (j & 1) ? hi(L::pair(ru, j >> 1)) : lo(L::pair(ru, j >> 1));
            const float* rb = cB + (g + j) * NT;
#pragma unroll
            for (int q = 0; q < NP; q += 2) {
              const float4 bv = *reinterpret_cast<const float4*>(rb + 2 * q);
              local_pair<ZOH>(acc[q], wc[q], A2[q], iA2[q], R, dt, du, uu, pk(bv.x, bv.y));
              local_pair<ZOH>(acc[q + 1], wc[q + 1], A2[q + 1], iA2[q + 1], R, dt, du, uu, pk(bv.z, bv.w));
            }
            R += dt;
          }
        } else {
          const int nv = min(kGroup, tn - g);
          for (int j = nv - 1; j >= 0; --j) {
            const int64_t ix = w.row + t + j;
            const float x = L::one(a.delta, ix) + bias;
            const float dt = a.softplus ? softplus(x) : x;
            const float du = dt * L::one(a.u, ix);
            const float uu = L::one(a.u, ix);
            const float* rb = cB + (g + j) * NT;
#pragma unroll
            for (int q = 0; q < NP; ++q) {
              const f2 bq = *reinterpret_cast<const f2*>(rb + 2 * q);
              local_pair<ZOH>(acc[q], wc[q], A2[q], iA2[q], R, dt, du, uu, bq);
            }
            R += dt;
          }
        }
      }
    }
    // Every weight left in this chunk underflows for every channel of the block: stop.
    const bool dead = !w.active || (may_stop && amax * R < kDead);
    if (__syncthreads_and(dead)) break;
    if (more) {
      segB.store(sB[buf ^ 1], sn, tseg);
      __syncthreads();
      buf ^= 1;
    }
  }

  cp_async_wait<0>();
  if (!w.active) return;
  a.ws_S[w.k * a.batch * a.dim + w.bd] = R;
  float* H = a.ws_H + (w.k * a.batch * a.dim + w.bd) * N;
#pragma unroll
  for (int q = 0; q < NP; ++q) {
    if (2 * q < N) H[2 * q] = lo(acc[q]);
    if (2 * q + 1 < N) H[2 * q + 1] = hi(acc[q]);
  }
}

}  // namespace ssk
