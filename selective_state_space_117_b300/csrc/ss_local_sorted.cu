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
// Data movement: a warp is its own block (no block barriers).  Its 32 channels are rows scattered
// over the (batch * dim, L) arrays, so one lane gathers each 16-step tile of their u and delta rows
// with tensor-memory-accelerator gathers (cp.async.bulk.tensor ... tile::gather4: four rows by
// index per instruction, eight per array) and the tile's B rows with one 3-D tensor load, all
// completing on the slot's mbarrier; a ring of kLsSlots tiles keeps the copies ahead.  (Per-lane
// 16-byte copies from 32 different rows cost 32 L1 requests per instruction, and the memory
// instruction queue, not the arithmetic, then bounded the pass.)  bf16 B rows are widened once
// per tile into an fp32 [state][step] tile that every lane reads as broadcast 16-byte loads.  Per
// state and pair of steps: one packed multiply for the exponent, two MUFU.EX2, one packed multiply
// for the input term, one packed fma.  Every wait on an mbarrier is bounded; a wait that gives up
// stops the warp (no further copy is issued) after the copies in flight have landed.
#include <type_traits>

#include "ss_kernels.cuh"
#include "ss_launch.h"
#include "ss_tma.cuh"
#include "ss_tma_launch.cuh"

namespace ssk {

namespace {

constexpr int kLsSteps = 16;           // steps per tile
constexpr int kLsSlots = 4;            // tiles in flight per warp
// Warps per SM the register budget is set for (1-warp blocks).  Measured on the long sequence:
// 12 ran the pass in 0.775 ms, 16 in 0.80 (fewer registers), 8 and 10 no faster than 12; ring
// depths of 3 to 8 tiles and 32-step tiles changed nothing.
constexpr int kLsMinBlocks = 12;
constexpr int kBuckets = 64;
constexpr unsigned kFull = 0xffffffffu;
constexpr float kDeadArg = -127.f;     // ex2 of anything below is under 2^-127: 0 after flushing

// Speed bucket of channel d: the slowest state's decay per step at the typical step size,
// softplus(bias) * min_n(-A[d, n]), on a log scale (2 buckets per octave, slowest first).  A
// channel with a state that does not decay (-A <= 0) goes to bucket 0.  The A row is read with
// independent loads (16-byte ones when the row allows), so their latencies overlap.
__device__ __forceinline__ int speed_bucket(const ScanArgs& a, int64_t d) {
  const int N = (int)a.dstate;
  const float* row = a.A + d * N;
  float rate = INFINITY;
  if ((N & 3) == 0 && (reinterpret_cast<uintptr_t>(row) & 15) == 0) {
    const float4* r4 = reinterpret_cast<const float4*>(row);
#pragma unroll 4
    for (int q = 0; q < N / 4; ++q) {
      const float4 v = __ldg(r4 + q);
      rate = fminf(rate, fminf(fminf(-v.x, -v.y), fminf(-v.z, -v.w)));
    }
  } else {
#pragma unroll 4
    for (int n = 0; n < N; ++n) rate = fminf(rate, -__ldg(row + n));
  }
  if (!(rate > 0.f)) return 0;
  const float key = softplus(a.delta_bias ? __ldg(a.delta_bias + d) : 0.f) * rate;
  if (!(key > 0.f)) return 0;
  const int b = (int)floorf(__log2f(key) * 2.f) + 48;
  return min(max(b, 1), kBuckets - 1);
}

// Channels whose buckets the order kernel keeps in shared memory between its two passes (beyond
// this, the second pass computes them again).
constexpr int kOrderSmem = 32768;

// perm[0 .. dim) = the channels in increasing speed bucket (one block): count the buckets, take
// the running sums, then place every channel.
__global__ void __launch_bounds__(1024) order_channels_kernel(const ScanArgs a, int* perm) {
  __shared__ int cnt[kBuckets];
  __shared__ unsigned char sb[kOrderSmem];
  const int tid = threadIdx.x;
  const bool keep = a.dim <= kOrderSmem;
  if (tid < kBuckets) cnt[tid] = 0;
  __syncthreads();
  for (int64_t d = tid; d < a.dim; d += blockDim.x) {
    const int bk = speed_bucket(a, d);
    if (keep) sb[d] = (unsigned char)bk;
    atomicAdd(&cnt[bk], 1);
  }
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
  for (int64_t d = tid; d < a.dim; d += blockDim.x) {
    const int pos = atomicAdd(&cnt[keep ? sb[d] : speed_bucket(a, d)], 1);
    if (span_ok(a.err, pos, 1, a.dim)) perm[pos] = (int)d;
  }
}

// Tensor maps of one call: u and delta as 2-D (L, batch * dim) arrays gathered by row, B as the
// 3-D (L, N, batch) array of the other TMA kernels.
struct LsMaps {
  CUtensorMap u, delta, B;
};

constexpr int align128(int x) { return (x + 127) / 128 * 128; }

template <int NT, bool BF>
struct LsLayout {
  static constexpr int ES = In<BF>::kBytes;
  static constexpr int RB = kLsSteps * ES;     // bytes of one row of a tile: 32 (bf16) or 64 (fp32)
  static constexpr int kIn = 32 * RB;          // u or delta rows of the warp's 32 channels, [lane][RB]
  static constexpr int kB = NT * RB;           // the tile's raw B rows, [state][step]
  static constexpr int kSlot = align128(2 * kIn + kB);
  static constexpr int kBf = BF ? NT * kLsSteps * 4 : 0;   // B widened to fp32 (bf16 inputs)
  static constexpr int oBf = kLsSlots * kSlot;
  static constexpr int oRows = oBf + kBf;      // the warp's 32 row indices (b * dim + d)
  static constexpr int oBar = oRows + 128;
  static constexpr int kBytes = oBar + kLsSlots * 8;
  static constexpr int kBPieces = NT * (RB / 16);   // 16-byte pieces of raw B per tile
};

// Gather of the 16-byte-aligned (x, rows r.x .. r.w) box of a 2-D tensor map: four rows of the
// map's box width land one after the other at dst, completing on bar.
__device__ __forceinline__ void tma_gather4(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int4 r) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(r.x), "r"(r.y), "r"(r.z), "r"(r.w), "r"(smem_addr(bar))
      : "memory");
}

// A lane's row of a tile (kLsSteps steps, RB bytes at lane * RB) as pairs of steps.
template <bool BF>
__device__ __forceinline__ void row_pairs(const unsigned char* arr, int lane, f2 (&v)[kLsSteps / 2]) {
  const unsigned char* row = arr + lane * kLsSteps * In<BF>::kBytes;
  if constexpr (BF) {
#pragma unroll
    for (int c = 0; c < kLsSteps / 8; ++c) {
      const uint4 r = *reinterpret_cast<const uint4*>(row + c * 16);
      v[4 * c] = bf16x2(r.x);
      v[4 * c + 1] = bf16x2(r.y);
      v[4 * c + 2] = bf16x2(r.z);
      v[4 * c + 3] = bf16x2(r.w);
    }
  } else {
#pragma unroll
    for (int c = 0; c < kLsSteps / 4; ++c) {
      const float4 r = *reinterpret_cast<const float4*>(row + c * 16);
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
__global__ void __launch_bounds__(32, kLsMinBlocks)
    local_sorted_kernel(const ScanArgs a, const int* __restrict__ perm, int64_t kchunks,
                        const __grid_constant__ LsMaps m) {
  using Lay = LsLayout<NT, BF>;
  constexpr int S = kLsSlots;
  constexpr int NPAIR = kLsSteps / 2;
  __shared__ __align__(128) unsigned char sm[Lay::kBytes];
  int* rows = reinterpret_cast<int*>(sm + Lay::oRows);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + Lay::oBar);

  const int lane = threadIdx.x;
  const int64_t items_per_group = a.batch * kchunks;
  const int64_t g = blockIdx.x / items_per_group, rem = blockIdx.x % items_per_group;
  const int64_t b = rem / kchunks, k = rem % kchunks;
  const int N = (int)a.dstate;
  const int64_t slot = g * 32 + lane;
  const int64_t BD = a.batch * a.dim;
  bool active = slot < a.dim;
  int64_t d = perm[active ? slot : a.dim - 1];
  const int64_t t_begin = k * a.chunk_len;
  const int ntiles = (int)(a.chunk_len / kLsSteps);   // the launcher guarantees whole tiles
  // Debug build: the channel, its rows of u/delta and B, its A row and workspace entries.
  if (!span_ok(a.err, d, 1, a.dim)) d = 0, active = false;
  const int64_t bd = b * a.dim + d;
  {
    const int64_t N = a.dstate;
    bool inb = span_ok(a.err, bd * a.seqlen + t_begin, a.chunk_len, BD * a.seqlen);
    inb = span_ok(a.err, b * N * a.seqlen + t_begin, (N - 1) * a.seqlen + a.chunk_len, a.batch * N * a.seqlen) && inb;
    inb = span_ok(a.err, (k * BD + bd) * N, N, a.nchunks * BD * N) && span_ok(a.err, k, 1, a.nchunks) && inb;
    active = active && inb;
  }

  // Per-state constants: A' = A * log2(e) (0 for padding states, which are never processed),
  // and each group's slowest A' (the last of its states to die).
  constexpr int NG = (NT + kLsGroup - 1) / kLsGroup;
  float Ap[NT], iAs[NT], gmax[NG];
#pragma unroll
  for (int gi = 0; gi < NG; ++gi) gmax[gi] = -INFINITY;
#pragma unroll
  for (int n = 0; n < NT; ++n) {
    const float an = (n < N) ? a.A[d * N + n] : 0.f;
    Ap[n] = an * kLog2e;
    iAs[n] = an != 0.f ? 1.f / an : 0.f;
    if (n < N) gmax[n / kLsGroup] = fmaxf(gmax[n / kLsGroup], Ap[n]);
  }
  const float bias = a.delta_bias ? a.delta_bias[d] : 0.f;
  const f2 bias2 = pk(bias, bias);
  const bool may_stop = a.softplus != 0;

  // Raw B rows of padding states stay zero in every slot; the warp's row indices; the barriers.
#pragma unroll
  for (int q0 = 0; q0 < Lay::kBPieces; q0 += 32) {
    const int q = q0 + lane;
    if (q < Lay::kBPieces && q / (Lay::RB / 16) >= N)
      for (int s = 0; s < S; ++s)
        *reinterpret_cast<uint4*>(sm + s * Lay::kSlot + 2 * Lay::kIn + q * 16) = make_uint4(0, 0, 0, 0);
  }
  rows[lane] = (int)bd;
  if (lane == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&bar[s], 1);
    mbar_init_fence();
  }
  __syncwarp();

  // Lane 0: copies of time tile (ntiles - 1 - i) into ring slot i % S (the walk goes backward).
  auto issue = [&](int i) {
    unsigned char* s = sm + (i % S) * Lay::kSlot;
    uint64_t* br = &bar[i % S];
    mbar_expect_tx(br, 2 * Lay::kIn + N * Lay::RB);
    const int x = (int)(t_begin + (int64_t)(ntiles - 1 - i) * kLsSteps);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int4 r4 = *reinterpret_cast<const int4*>(rows + 4 * j);
      tma_gather4(s + j * 4 * Lay::RB, &m.u, br, x, r4);
      tma_gather4(s + Lay::kIn + j * 4 * Lay::RB, &m.delta, br, x, r4);
    }
    tma_load_3d(s + 2 * Lay::kIn, &m.B, br, x, 0, (int)b);
  };
  int issued = 0;   // tiles whose copies lane 0 has issued
  if (lane == 0) {
    prefetch_tensormap(&m.u);
    prefetch_tensormap(&m.delta);
    prefetch_tensormap(&m.B);
  }
  for (int i = 0; i < S - 1 && i < ntiles; ++i) {
    if (lane == 0) issue(i);
    issued = i + 1;
  }

  f2 acc[NT];
#pragma unroll
  for (int n = 0; n < NT; ++n) acc[n] = pk(0.f, 0.f);
  float R = 0.f;   // sum of dt after the current tile
  bool ok = true;
  int i = 0;

  for (; i < ntiles; ++i) {
    // The groups with a state whose weights have not underflowed in some channel of the warp
    // (all votes first: they depend only on R, not on this tile's data).  None left: the rest
    // of the chunk adds zeros.
    const float R_in = R;
    unsigned live = 0;
#pragma unroll
    for (int gi = 0; gi < NG; ++gi)
      if (gi * kLsGroup < N && (!may_stop || __any_sync(kFull, active && gmax[gi] * R_in >= kDeadArg)))
        live |= 1u << gi;
    if (live == 0) break;
    if (i + S - 1 < ntiles) {   // into the slot of tile i - 1, which every lane has finished with
      if (lane == 0) issue(i + S - 1);
      issued = i + S;
    }
    ok = __all_sync(kFull, mbar_wait(&bar[i % S], (i / S) & 1, a.err));
    if (!ok) break;
    const unsigned char* s = sm + (i % S) * Lay::kSlot;
    const float* Bt;
    if constexpr (BF) {
      // Widen the tile's B rows to fp32: lane q converts piece q (8 steps of one state).
      float* bf = reinterpret_cast<float*>(sm + Lay::oBf);
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
    // after[p] = sum of dt over the pairs after p in the tile (sums of pairs first, then a chain).
    {
      float ps[NPAIR], after[NPAIR];
#pragma unroll
      for (int p = 0; p < NPAIR; ++p) ps[p] = lo(dt2[p]) + hi(dt2[p]);
      after[NPAIR - 1] = 0.f;
#pragma unroll
      for (int p = NPAIR - 2; p >= 0; --p) after[p] = after[p + 1] + ps[p + 1];
#pragma unroll
      for (int p = 0; p < NPAIR; ++p) {
        const float r_hi = R_in + after[p];
        R2[p] = pk(r_hi + hi(dt2[p]), r_hi);
      }
      R = R_in + (ps[0] + after[0]);
    }

    // One state of the tile: its terms for the 16 steps added to acc[n].
    auto state_tile = [&](int n) {
      const float4* brow = reinterpret_cast<const float4*>(Bt + n * kLsSteps);
      const f2 A2 = pk(Ap[n], Ap[n]);
      f2 sum = acc[n];
      if constexpr (ZOH) {
        // Weights at the points R_{-1} = R (before the tile), R_0, ..., R_{kLsSteps-1}: the hold
        // weight of step s is (w(R_{s-1}) - w(R_s)) / A with w(R) = exp(A R).
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
    };
#pragma unroll
    for (int gi = 0; gi < NG; ++gi) {
      if (!((live >> gi) & 1u)) continue;
      if constexpr (ZOH) {
        // With the hold a state's tile is a long stretch of code; unrolled over the group's
        // states it overflowed the instruction cache (ncu: a warp per issue waiting for
        // instructions), so this loop stays rolled (its per-state constants come from local
        // memory): the long-sequence ZOH local pass 1.33 -> 1.20 ms.
#pragma unroll 1
        for (int n = gi * kLsGroup; n < (gi + 1) * kLsGroup && n < N; ++n) state_tile(n);
      } else {
#pragma unroll
        for (int n = gi * kLsGroup; n < (gi + 1) * kLsGroup && n < NT; ++n) {
          if (n >= N) break;
          state_tile(n);
        }
      }
    }
    __syncwarp();   // every lane is done with this slot and the fp32 B tile before they are refilled
  }
  // Tiles i .. issued - 1 were issued and not waited for (after an early stop, or the tile whose
  // wait gave up): wait for each (bounded; a completed phase returns at once) before exiting.
  if (lane == 0)
    for (int j = i; j < issued; ++j) mbar_wait(&bar[j % S], (j / S) & 1, nullptr);
  __syncwarp();

  if (!active || !ok) return;
  a.ws_S[k * BD + bd] = R;
  float* H = a.ws_H + (k * BD + bd) * N;
#pragma unroll
  for (int n = 0; n < NT; ++n)
    if (n < N) H[n] = lo(acc[n]) + hi(acc[n]);
}

// (L, rows) row-major array as a 2-D tensor map gathered one row at a time (box: kLsSteps x 1).
inline bool encode_rows(CUtensorMap* mp, bool bf16, const void* base, int64_t L, int64_t rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const int64_t es = bf16 ? 2 : 4;
  cuuint64_t dims[2] = {(cuuint64_t)L, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(L * es)};
  cuuint32_t box[2] = {(cuuint32_t)kLsSteps, 1};
  cuuint32_t estr[2] = {1, 1};
  return fn(mp, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base),
            dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int NT, bool BF, bool ZOH>
int go_local_sorted(const ScanArgs& a, int64_t kchunks, cudaStream_t s) {
  LsMaps m;
  const int64_t rows = a.batch * a.dim;
  if (!encode_rows(&m.u, BF, a.u, a.seqlen, rows) || !encode_rows(&m.delta, BF, a.delta, a.seqlen, rows) ||
      !encode3d(&m.B, BF, false, a.B, a.seqlen, a.dstate, a.batch, kLsSteps, (unsigned)a.dstate,
                CU_TENSOR_MAP_SWIZZLE_NONE))
    return 1;
  const int64_t groups = (a.dim + 31) / 32;
  const int64_t items = groups * a.batch * kchunks;
  order_channels_kernel<<<1, 1024, 0, s>>>(a, a.perm);
  local_sorted_kernel<NT, BF, ZOH><<<(unsigned)items, 32, 0, s>>>(a, a.perm, kchunks, m);
  return 0;
}

}  // namespace

bool local_sorted_available(const ScanArgs& a, bool bf16) {
  (void)bf16;
  const int64_t kchunks = a.local_chunks;
  if (kchunks < 1 || !a.perm || !encode_fn()) return false;
  if (a.dstate < 1 || a.dstate > 16 || !a.vec || !a.vec_bc || a.chunk_len % kLsSteps != 0) return false;
  if (a.batch * a.dim > (int64_t)INT32_MAX || a.seqlen > (int64_t)INT32_MAX) return false;
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
