// Forward scan with TMA-staged inputs and outputs (sm_103a).
//
// Same work decomposition and arithmetic as scan_kernel (one thread per
// (batch row, channel, chunk), states in registers, scan_group for every 8
// steps), but every operand moves as a bulk tensor copy: per 16-step tile one
// thread issues 3-D TMA loads of the block's u, delta and z rows (swizzled, so
// each thread's row reads are bank-conflict free) and of B_t and C_t, into a
// ring of kTmaSlots tiles completed by mbarriers, and one bulk tensor store
// writes the block's 64 x 16 tile of y.  The threads do no per-element global
// address arithmetic and issue no scattered loads or stores.
#pragma once

#include "ss_kernels.cuh"
#include "ss_tma.cuh"

namespace ssk {

constexpr int kTmaSteps = 16;  // steps per tile
constexpr int kTmaSlots = 3;   // input tiles in flight

struct alignas(64) TmaMaps {
  CUtensorMap u, delta, z, B, C, y;
};

constexpr int align1k(int x) { return (x + 1023) / 1024 * 1024; }

// Shared-memory layout (byte offsets from a 1024-byte aligned base).
template <int NT, bool BF, bool HAS_Z>
struct TmaLayout {
  static constexpr int ES = In<BF>::kBytes;
  static constexpr int RB = kTmaSteps * ES;   // input row bytes: 32 (bf16) or 64 (fp32) = swizzle span
  static constexpr int YB = kTmaSteps * 4;    // y row bytes: 64 = swizzle span
  static constexpr int NA = HAS_Z ? 3 : 2;
  static constexpr int kIn = kCh * RB;        // one input array's tile
  static constexpr int kBC = NT * RB;         // one raw B or C tile (N <= NT rows)
  static constexpr int kSlot = align1k(NA * kIn + 2 * kBC);
  static constexpr int kY = kCh * YB;
  static constexpr int kBCf = kTmaSteps * NT * 4;  // one fp32 B or C tile, [t][n]
  static constexpr int oY = kTmaSlots * kSlot;
  static constexpr int oBCf = oY + 2 * kY;
  static constexpr int oBar = oBCf + 4 * kBCf;
  static constexpr int kBytes = oBar + kTmaSlots * 8;
  static constexpr int kAlloc = kBytes + 1024;   // slack to align the base
};

// Thread 0: load tile k (inputs and B/C) into its slot and arm the slot's barrier.
template <int NT, bool BF, bool HAS_Z>
__device__ __forceinline__ void tma_issue(const TmaMaps& m, unsigned char* sm, uint64_t* bar, int k, int64_t t_begin,
                                          int y0, int zb, int N) {
  using Lay = TmaLayout<NT, BF, HAS_Z>;
  const int s = k % kTmaSlots;
  unsigned char* slot = sm + s * Lay::kSlot;
  mbar_expect_tx(&bar[s], Lay::NA * Lay::kIn + 2 * N * Lay::RB);
  const int x = (int)(t_begin + (int64_t)k * kTmaSteps);
  tma_load_3d(slot, &m.u, &bar[s], x, y0, zb);
  tma_load_3d(slot + Lay::kIn, &m.delta, &bar[s], x, y0, zb);
  if (HAS_Z) tma_load_3d(slot + 2 * Lay::kIn, &m.z, &bar[s], x, y0, zb);
  tma_load_3d(slot + Lay::NA * Lay::kIn, &m.B, &bar[s], x, 0, zb);
  tma_load_3d(slot + Lay::NA * Lay::kIn + Lay::kBC, &m.C, &bar[s], x, 0, zb);
}

// All threads: NARR raw [n][t] tiles (B, then C; N rows of RB bytes, NT rows
// apart) starting at `raw` into fp32 [t][n] tiles of NT columns at dst[0..]
// (zero for n >= N).
template <int NT, bool BF, int NARR>
__device__ __forceinline__ void tma_convert_rows(const unsigned char* raw, int N, float* const (&dst)[NARR], int tid) {
  using L = In<BF>;
  constexpr int ES = L::kBytes;
  constexpr int RB = kTmaSteps * ES;
  constexpr int SEGS = kTmaSteps / kGroup;
  const unsigned base = smem_addr(raw);
  for (int e = tid; e < NARR * NT * SEGS; e += kCh) {
    const int arr = e / (NT * SEGS), rem = e % (NT * SEGS), n = rem % NT, q = rem / NT;
    float v[kGroup];
    if (n < N) {
      const typename L::Raw8 r = L::from_smem(base + (arr * NT + n) * RB + q * kGroup * ES, 16);
#pragma unroll
      for (int p = 0; p < kGroup / 2; ++p) {
        const f2 x = L::pair(r, p);
        v[2 * p] = lo(x);
        v[2 * p + 1] = hi(x);
      }
    } else {
#pragma unroll
      for (int j = 0; j < kGroup; ++j) v[j] = 0.f;
    }
    float* d = dst[arr];
#pragma unroll
    for (int j = 0; j < kGroup; ++j) d[(q * kGroup + j) * NT + n] = v[j];
  }
}

template <int NT, bool BF, bool HAS_Z>
__device__ __forceinline__ void tma_convert_bc(const unsigned char* slot, int N, float* dB, float* dC, int tid) {
  using Lay = TmaLayout<NT, BF, HAS_Z>;
  float* const dst[2] = {dB, dC};
  tma_convert_rows<NT, BF, 2>(slot + Lay::NA * Lay::kIn, N, dst, tid);
}

template <int NT, bool BF, bool HAS_Z, int MODE, bool ZOH>
__global__ void __launch_bounds__(kCh, (MinBlocks<NT, BF>::value))
    scan_tma_kernel(const ScanArgs a, const __grid_constant__ TmaMaps m) {
  using L = In<BF>;
  using Lay = TmaLayout<NT, BF, HAS_Z>;
  constexpr int NP = NT / 2;
  constexpr int TS = kTmaSteps;
  constexpr int S = kTmaSlots;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + Lay::oBar);

  const int tid = threadIdx.x;
  Unit w = unit_of(a);
  w.active = w.active && unit_ok(a, w);
  const int N = (int)a.dstate;
  const int ct = blockIdx.x % a.ctiles;
  const int ntiles = (int)((w.t_end - w.t_begin + TS - 1) / TS);
  const int y0 = ct * kCh, zb = (int)w.b;

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

  if (tid == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&bar[s], 1);
    mbar_init_fence();
  }
  __syncthreads();
  if (tid == 0)
    for (int k = 0; k < S && k < ntiles; ++k) tma_issue<NT, BF, HAS_Z>(m, sm, bar, k, w.t_begin, y0, zb, N);

  float* bcf = reinterpret_cast<float*>(sm + Lay::oBCf);  // [buffer][B, C][TS * NT]
  constexpr int BCF = Lay::kBCf / 4;
  // Every thread waits on the tile's barrier itself; the block then agrees on the
  // outcome at the barrier that follows (__syncthreads_and), so that once any wait
  // has given up no thread computes on the tile and thread 0 starts no further
  // load or store.  Loads already in flight are then waited for (bounded) below.
  bool ok = mbar_wait(&bar[0], 0, a.err);
  tma_convert_bc<NT, BF, HAS_Z>(sm, N, bcf, bcf + BCF, tid);
  ok = __syncthreads_and(ok);
  int pending = 0;                 // on a failure: the first tile whose load may still be in flight
  int issued = min(S, ntiles);     // tiles whose loads thread 0 has issued

  for (int k = 0; ok && k < ntiles; ++k) {
    const int s = k % S;
    const unsigned slot = smem_addr(sm + s * Lay::kSlot);
    unsigned char* yt = sm + Lay::oY + (k & 1) * Lay::kY;
    const float* cB = bcf + (k & 1) * 2 * BCF;
    const float* cC = cB + BCF;
    const int64_t t0 = w.t_begin + (int64_t)k * TS;
    if (w.active) {
      const unsigned ybase = smem_addr(yt);
      // With the zero-order hold one 8-step group is already a long stretch of code; unrolling
      // the tile's two groups as well overflowed the instruction cache (ncu: a warp per issue
      // waiting for instructions) and cost 5.6% of the long-sequence fix-up.
#pragma unroll(ZOH ? 1 : TS / kGroup)
      for (int g = 0; g < TS / kGroup; ++g) {
        if (t0 + g * kGroup >= w.t_end) break;
        const typename L::Raw8 cu = tile_row8<BF, Lay::RB>(slot, tid, g);
        const typename L::Raw8 rd = tile_row8<BF, Lay::RB>(slot + Lay::kIn, tid, g);
        typename L::Raw8 cz{};
        if (HAS_Z) cz = tile_row8<BF, Lay::RB>(slot + 2 * Lay::kIn, tid, g);
        f2 y2[4];
        scan_group<NT, BF, HAS_Z, ZOH, MODE == kFull>(cu, rd, cz, bias2, D2, a.softplus, A2, iA2, h,
                                                      cB + g * kGroup * NT, cC + g * kGroup * NT, y2);
        sts16(ybase + swz<Lay::YB>(tid, 2 * g), make_float4(lo(y2[0]), hi(y2[0]), lo(y2[1]), hi(y2[1])));
        sts16(ybase + swz<Lay::YB>(tid, 2 * g + 1), make_float4(lo(y2[2]), hi(y2[2]), lo(y2[3]), hi(y2[3])));
      }
    }
    fence_async_smem();
    if (k + 1 < ntiles) {
      const int s1 = (k + 1) % S;
      ok = mbar_wait(&bar[s1], ((k + 1) / S) & 1, a.err);
      float* nb = bcf + ((k + 1) & 1) * 2 * BCF;
      tma_convert_bc<NT, BF, HAS_Z>(sm + s1 * Lay::kSlot, N, nb, nb + BCF, tid);
    }
    if (tid == 0) bulk_wait_read<0>();  // the previous tile's y store has left the other buffer
    ok = __syncthreads_and(ok);
    if (!ok) {
      pending = k + 1;
      break;
    }
    if (tid == 0) {
      tma_store_3d(&m.y, yt, (int)t0, y0, zb);
      bulk_commit();
      if (k + S < ntiles) {
        tma_issue<NT, BF, HAS_Z>(m, sm, bar, k + S, w.t_begin, y0, zb, N);
        issued = k + S + 1;
      }
    }
  }
  if (tid == 0) {
    // After a failure, tiles pending .. issued - 1 were issued and not all seen to land: wait
    // for each (bounded; a completed phase returns at once) before the block exits.
    if (!ok)
      for (int j = pending; j < issued; ++j) mbar_wait(&bar[j % S], (j / S) & 1, nullptr);
    bulk_wait_read<0>();   // the y tiles have been read out of shared memory; their writes complete on their own
  }

  // The final state: after the whole sequence, or after the last chunk of the chunked scan.
  if ((MODE == kFull || w.k == a.nchunks - 1) && w.active && ok && a.last_state) {
    float* out = a.last_state + w.bd * N;
#pragma unroll
    for (int q = 0; q < NP; ++q) {
      if (2 * q < N) out[2 * q] = lo(h[q]);
      if (2 * q + 1 < N) out[2 * q + 1] = hi(h[q]);
    }
  }
}

// Shared-memory layout of local_tma_kernel: slots of (u, delta, raw B).
template <int NT, bool BF>
struct LocalTmaLayout {
  static constexpr int ES = In<BF>::kBytes;
  static constexpr int RB = kTmaSteps * ES;
  static constexpr int kIn = kCh * RB;
  static constexpr int kBC = NT * RB;
  static constexpr int kSlot = align1k(2 * kIn + kBC);
  static constexpr int kBf = kTmaSteps * NT * 4;
  static constexpr int oBf = kTmaSlots * kSlot;
  static constexpr int oBar = oBf + 2 * kBf;
  static constexpr int kBytes = oBar + kTmaSlots * 8 + 8;   // barriers, then the failure flag
  static constexpr int kAlloc = kBytes + 1024;
};

// The chunked scan's local pass (see local_kernel for the computation and its
// early stop) with TMA-staged inputs: tiles are loaded and consumed from the
// chunk's end backward.  A block that stops early first waits for the loads
// it has already issued, so no bulk copy lands in shared memory after exit.
template <int NT, bool BF, bool ZOH>
__global__ void __launch_bounds__(kCh, (MinBlocks<NT, BF>::value))
    local_tma_kernel(const ScanArgs a, const __grid_constant__ TmaMaps m) {
  using L = In<BF>;
  using Lay = LocalTmaLayout<NT, BF>;
  constexpr int NP = NT / 2;
  constexpr int TS = kTmaSteps;
  constexpr int S = kTmaSlots;
  constexpr float kDead = -127.f;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + Lay::oBar);

  const int tid = threadIdx.x;
  Unit w = unit_of(a);
  w.active = w.active && unit_ok(a, w);
  const int N = (int)a.dstate;
  const int ct = blockIdx.x % a.ctiles;
  const int ntiles = (int)((w.t_end - w.t_begin + TS - 1) / TS);
  const int y0 = ct * kCh, zb = (int)w.b;

  f2 A2[NP], iA2[NP], wc[NP], acc[NP];
  float amax = -1e30f;
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

  // Tile k of the loop is time tile ntiles - 1 - k of the chunk.
  auto issue = [&](int k) {
    const int s = k % S;
    unsigned char* slot = sm + s * Lay::kSlot;
    mbar_expect_tx(&bar[s], 2 * Lay::kIn + N * Lay::RB);
    const int x = (int)(w.t_begin + (int64_t)(ntiles - 1 - k) * TS);
    tma_load_3d(slot, &m.u, &bar[s], x, y0, zb);
    tma_load_3d(slot + Lay::kIn, &m.delta, &bar[s], x, y0, zb);
    tma_load_3d(slot + 2 * Lay::kIn, &m.B, &bar[s], x, 0, zb);
  };
  if (tid == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&bar[s], 1);
    *reinterpret_cast<int*>(sm + Lay::oBar + kTmaSlots * 8) = 0;
    mbar_init_fence();
  }
  __syncthreads();
  if (tid == 0)
    for (int k = 0; k < S && k < ntiles; ++k) issue(k);

  float* bf = reinterpret_cast<float*>(sm + Lay::oBf);
  constexpr int BF_ = Lay::kBf / 4;
  // A wait that gives up raises s_fail before the tile's barrier; after the barrier
  // every thread sees it, the block stops, and thread 0 waits (bounded) for the loads
  // still in flight before the block exits, as on an early stop.
  int* s_fail = reinterpret_cast<int*>(sm + Lay::oBar + kTmaSlots * 8);
  bool ok = mbar_wait(&bar[0], 0, a.err);
  {
    float* const d0[1] = {bf};
    tma_convert_rows<NT, BF, 1>(sm + 2 * Lay::kIn, N, d0, tid);
  }
  if (!ok) *s_fail = 1;
  __syncthreads();
  ok = *s_fail == 0;
  int pending = ok ? ntiles : 0;   // the first tile whose load may still be in flight
  int issued = min(S, ntiles);     // tiles whose loads thread 0 has issued

  for (int k = 0; ok && k < ntiles; ++k) {
    const int s = k % S;
    const unsigned slot = smem_addr(sm + s * Lay::kSlot);
    const float* cB = bf + (k & 1) * BF_;
    const int64_t t0 = w.t_begin + (int64_t)(ntiles - 1 - k) * TS;
    if (w.active) {
#pragma unroll
      for (int g = TS / kGroup - 1; g >= 0; --g) {
        if (t0 + g * kGroup >= w.t_end) continue;
        const typename L::Raw8 ru = tile_row8<BF, Lay::RB>(slot, tid, g);
        const typename L::Raw8 rd = tile_row8<BF, Lay::RB>(slot + Lay::kIn, tid, g);
        f2 dt2[4], du2[4];
        step_scalars<BF>(ru, rd, bias2, a.softplus, dt2, du2);
#pragma unroll
        for (int j = kGroup - 1; j >= 0; --j) {
          const float dt = (j & 1) ? hi(dt2[j >> 1]) : lo(dt2[j >> 1]);
          const float du = (j & 1) ? hi(du2[j >> 1]) : lo(du2[j >> 1]);
          const float uu = (j & 1) ? hi(L::pair(ru, j >> 1)) : lo(L::pair(ru, j >> 1));
          const float* rb = cB + (g * kGroup + j) * NT;
#pragma unroll
          for (int q = 0; q < NP; q += 2) {
            const float4 bv = *reinterpret_cast<const float4*>(rb + 2 * q);
            local_pair<ZOH>(acc[q], wc[q], A2[q], iA2[q], R, dt, du, uu, pk(bv.x, bv.y));
            local_pair<ZOH>(acc[q + 1], wc[q + 1], A2[q + 1], iA2[q + 1], R, dt, du, uu, pk(bv.z, bv.w));
          }
          R += dt;
        }
      }
    }
    if (k + 1 < ntiles) {
      const int s1 = (k + 1) % S;
      if (!mbar_wait(&bar[s1], ((k + 1) / S) & 1, a.err)) *s_fail = 1;
      float* const d1[1] = {bf + ((k + 1) & 1) * BF_};
      tma_convert_rows<NT, BF, 1>(sm + s1 * Lay::kSlot + 2 * Lay::kIn, N, d1, tid);
    }
    // Every weight left in this chunk underflows for every channel of the block: stop,
    // after the loads already issued (tiles k + 2 .. k + S - 1) have landed.
    const bool dead = !w.active || (may_stop && amax * R < kDead);
    const bool all_dead = __syncthreads_and(dead);
    if (*s_fail) {
      ok = false;
      pending = k + 1;
      break;
    }
    if (all_dead) {
      pending = k + 2;
      break;
    }
    if (k + S < ntiles) {
      if (tid == 0) issue(k + S);
      issued = k + S + 1;
    }
  }
  if (tid == 0)   // tiles pending .. issued - 1 may still be in flight (none after a full walk)
    for (int j = pending; j < issued; ++j) mbar_wait(&bar[j % S], (j / S) & 1, nullptr);

  if (!w.active || !ok) return;
  a.ws_S[w.k * a.batch * a.dim + w.bd] = R;
  float* H = a.ws_H + (w.k * a.batch * a.dim + w.bd) * N;
#pragma unroll
  for (int q = 0; q < NP; ++q) {
    if (2 * q < N) H[2 * q] = lo(acc[q]);
    if (2 * q + 1 < N) H[2 * q + 1] = hi(acc[q]);
  }
}

}  // namespace ssk
