// Launcher of the one-token decode step.
#include "ss_device.cuh"
#include "ss_dispatch.cuh"
#include "ss_launch.h"
#include "ss_tma.cuh"

namespace ssk {

// L2 cache policy for the state: the next step reads it again, so it is
// marked evict_last; the per-step inputs and y use the default policy.
// States per lane: 8 measured faster than 4 or 16 on B300 (42 vs 48 / 47 us
// per 256 x 5120 x 16 step): enough bytes in flight per thread without
// lowering the number of resident threads too far.
constexpr int kDecodeSpl = 8;

__device__ __forceinline__ uint64_t policy_keep() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ float4 ld_keep4(const float* p, uint64_t pol) {
  float4 v;
  asm volatile("ld.global.L2::cache_hint.v4.f32 {%0, %1, %2, %3}, [%4], %5;"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p), "l"(pol));
  return v;
}

__device__ __forceinline__ void st_keep4(float* p, float4 v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.v4.f32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p), "f"(v.x), "f"(v.y), "f"(v.z),
               "f"(v.w), "l"(pol)
               : "memory");
}

// The (x, y) block this block stands for: itself, or with `reverse` the block at the mirrored
// position of the grid's linear order, so that the state's ranges are taken last first.
__device__ __forceinline__ uint2 block_of(int reverse) {
  if (!reverse) return make_uint2(blockIdx.x, blockIdx.y);
  const unsigned n = gridDim.x * gridDim.y, lin = n - 1 - (blockIdx.y * gridDim.x + blockIdx.x);
  return make_uint2(lin % gridDim.x, lin / gridDim.x);
}

// One decode step.  A lane owns SPL = min(NT, kDecodeSpl) consecutive states of
// one channel (G = NT / SPL lanes per channel: 2 for N = 16), keeps them in
// registers as f32x2 pairs and reads and writes them as 16-byte vectors.  Grid:
// x covers the (channel, lane) pairs of one batch row, y is the batch row.
// Every load is issued before any arithmetic; with several lanes per channel
// each lane computes dt itself (no cross-lane wait) and the readout sum crosses
// the lanes with xor shuffles.
template <int NT, bool BF, bool HAS_Z, bool ZOH>
__global__ void __launch_bounds__(kDecodeThreads) decode_kernel(const DecodeArgs a, int reverse) {
  using L = In<BF>;
  constexpr int SPL = NT < kDecodeSpl ? NT : kDecodeSpl;
  constexpr int G = NT / SPL;
  constexpr int NP = SPL / 2;
  const uint2 blk = block_of(reverse);
  const int i = (int)blk.x * kDecodeThreads + threadIdx.x;
  const int d = i / G;
  const int l = i % G;
  if (d >= a.dim) return;                        // the lanes of a channel leave together
  const int N = (int)a.dstate;
  const int64_t b = blk.y;
  const int64_t c = b * a.dim + d;               // flattened (b, d)
  // Debug build: this channel's inputs, state row, A row and the batch row of B and C.
  if (!span_ok(a.err, c, 1, a.batch * a.dim) || !span_ok(a.err, c * N, N, a.batch * a.dim * N) ||
      !span_ok(a.err, (int64_t)d * N, N, a.dim * N) || !span_ok(a.err, b * N, N, a.batch * N))
    return;
  const int n0 = SPL * l;
  const uint64_t keep = policy_keep();

  // ---- loads
  const float x = L::one(a.delta, c) + (a.delta_bias ? a.delta_bias[d] : 0.f);
  const float uu = L::one(a.u, c);
  float zz = 0.f, Dd = 0.f;
  if (l == 0) {
    if (HAS_Z) zz = L::one(a.z, c);
    if (a.D) Dd = a.D[d];
  }
  float* st = a.state + c * N + n0;
  const float* Ar = a.A + (int64_t)d * N + n0;
  float hv[SPL], Av[SPL], Bv[SPL], Cv[SPL];
  if (a.vec) {                                   // N % 4 == 0, 16-byte state/A rows, 8-byte B/C rows
#pragma unroll
    for (int k = 0; k < SPL; k += 4) {
      if (n0 + k < N) {
        const float4 h4 = ld_keep4(st + k, keep);
        const float4 a4 = __ldg(reinterpret_cast<const float4*>(Ar + k));
        hv[k] = h4.x; hv[k + 1] = h4.y; hv[k + 2] = h4.z; hv[k + 3] = h4.w;
        Av[k] = a4.x; Av[k + 1] = a4.y; Av[k + 2] = a4.z; Av[k + 3] = a4.w;
        if (BF) {
          const uint2 b2 = __ldg(reinterpret_cast<const uint2*>(static_cast<const unsigned short*>(a.B) + b * N + n0 + k));
          const uint2 c2 = __ldg(reinterpret_cast<const uint2*>(static_cast<const unsigned short*>(a.C) + b * N + n0 + k));
          Bv[k] = bf16_lo(b2.x); Bv[k + 1] = bf16_hi(b2.x); Bv[k + 2] = bf16_lo(b2.y); Bv[k + 3] = bf16_hi(b2.y);
          Cv[k] = bf16_lo(c2.x); Cv[k + 1] = bf16_hi(c2.x); Cv[k + 2] = bf16_lo(c2.y); Cv[k + 3] = bf16_hi(c2.y);
        } else {
          const float4 b4 = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(a.B) + b * N + n0 + k));
          const float4 c4 = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(a.C) + b * N + n0 + k));
          Bv[k] = b4.x; Bv[k + 1] = b4.y; Bv[k + 2] = b4.z; Bv[k + 3] = b4.w;
          Cv[k] = c4.x; Cv[k + 1] = c4.y; Cv[k + 2] = c4.z; Cv[k + 3] = c4.w;
        }
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) hv[k + j] = Av[k + j] = Bv[k + j] = Cv[k + j] = 0.f;
      }
    }
  } else {
#pragma unroll
    for (int k = 0; k < SPL; ++k) {
      const bool ok = n0 + k < N;
      hv[k] = ok ? st[k] : 0.f;
      Av[k] = ok ? Ar[k] : 0.f;
      Bv[k] = ok ? L::one(a.B, b * N + n0 + k) : 0.f;
      Cv[k] = ok ? L::one(a.C, b * N + n0 + k) : 0.f;
    }
  }

  // ---- the step: dt, then every state pair, then the readout
  const float dt = a.softplus ? softplus(x) : x;
  const float du = dt * uu;
  const f2 dtp = pk(dt, dt), dup = pk(du, du), upp = pk(uu, uu), l2e = pk(kLog2e, kLog2e);
  f2 acc = pk(0.f, 0.f);
#pragma unroll
  for (int q = 0; q < NP; ++q) {
    const f2 hq = pk(hv[2 * q], hv[2 * q + 1]);
    const f2 Aq = pk(Av[2 * q], Av[2 * q + 1]);
    const f2 arg = mul2(dtp, mul2(l2e, Aq));
    const f2 e = ex2x2(arg);
    f2 hn;
    if constexpr (ZOH) {
      const f2 iA = pk(Av[2 * q] != 0.f ? 1.f / Av[2 * q] : 0.f, Av[2 * q + 1] != 0.f ? 1.f / Av[2 * q + 1] : 0.f);
      hn = fma2(e, hq, mul2(hold2(arg, e, dtp, iA), mul2(upp, pk(Bv[2 * q], Bv[2 * q + 1]))));
    } else {
      hn = fma2(e, hq, mul2(dup, pk(Bv[2 * q], Bv[2 * q + 1])));
    }
    hv[2 * q] = lo(hn);
    hv[2 * q + 1] = hi(hn);
    acc = fma2(pk(Cv[2 * q], Cv[2 * q + 1]), hn, acc);
  }
  float y = lo(acc) + hi(acc);

  // ---- stores
  if (a.vec) {
#pragma unroll
    for (int k = 0; k < SPL; k += 4)
      if (n0 + k < N) st_keep4(st + k, make_float4(hv[k], hv[k + 1], hv[k + 2], hv[k + 3]), keep);
  } else {
#pragma unroll
    for (int k = 0; k < SPL; ++k)
      if (n0 + k < N) st[k] = hv[k];
  }
  if (G > 1) {
    const int lane = threadIdx.x & 31;
    const unsigned gmask = ((1u << G) - 1u) << (lane & ~(G - 1));
#pragma unroll
    for (int off = G / 2; off > 0; off >>= 1) y += __shfl_xor_sync(gmask, y, off);
  }
  if (l == 0) {
    float yv = fmaf(Dd, uu, y);
    if (HAS_Z) yv *= silu(zz);
    a.y[c] = yv;
  }
}


// Untiled bulk copies (16-byte aligned addresses, sizes a multiple of 16) with an L2 policy.
__device__ __forceinline__ void bulk_load_hint(void* dst, const void* src, unsigned bytes, uint64_t* bar, uint64_t pol) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
               ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(pol) : "memory");
}
__device__ __forceinline__ void bulk_store_hint(void* dst, const void* src, unsigned bytes, uint64_t pol) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;"
               ::"l"(dst), "r"(smem_addr(src)), "r"(bytes), "l"(pol) : "memory");
}

// The same step with the block's slice of the state moved by one bulk copy each way:
// CPB consecutive channels of one batch row are one contiguous range of CPB * N floats
// (8 KB at N = 16).  One thread loads it into shared memory (completing on an
// mbarrier, with the state's evict_last L2 policy) while every thread loads its own
// inputs; the threads update their states in shared memory; one bulk store writes the
// range back.  Measured 38.2 us against 43.8 us per 256 x 5120 x 16 step (eager
// launches): the state moves with a few large copies instead of 16-byte loads and
// stores from every thread.  The wait on the mbarrier is bounded (mbar_wait records
// a timeout in the device status word); if any thread's wait gives up, the whole block
// skips the step, so the state is left unchanged and y is not written.
// With bf16 inputs the kernel is held to 32 registers, 8 blocks (64 warps) per SM: 32.4 us per
// 256 x 5120 x 16 step against 34.1 us at its own 36 registers and 6 blocks (a few bytes
// spilled; 45.8 against 46.5 us with the zero-order hold).  fp32 inputs keep the compiler's choice.
template <bool BF>
struct DecodeMinBlocks {
  static constexpr int value = BF ? 8 : 1;
};

template <int NT, bool BF, bool HAS_Z, bool ZOH>
__global__ void __launch_bounds__(kDecodeThreads, DecodeMinBlocks<BF>::value)
    decode_bulk_kernel(const DecodeArgs a, int reverse) {
  using L = In<BF>;
  constexpr int SPL = kDecodeSpl, G = NT / SPL, CPB = kDecodeThreads / G, NP = SPL / 2;
  __shared__ __align__(128) float sst[CPB * NT];
  // With the zero-order hold the block's A rows come with the state's copy (see below).
  __shared__ __align__(128) float sA[ZOH ? CPB * NT : 4];
  __shared__ __align__(8) uint64_t bar;
  const int tid = threadIdx.x;
  const uint2 blk = block_of(reverse);
  const int64_t b = blk.y, c0 = (int64_t)blk.x * CPB;
  const int nch = (int)min((int64_t)CPB, a.dim - c0);
  const int N = (int)a.dstate;
  const unsigned bytes = (unsigned)(nch * N * 4);
  float* gst = a.state + (b * a.dim + c0) * N;
  // Debug build: the block's contiguous range of the state, and the batch row of B and C (the
  // whole block leaves before any copy or barrier when one is outside).
  if (!span_ok(a.err, (b * a.dim + c0) * N, (int64_t)nch * N, a.batch * a.dim * N) ||
      !span_ok(a.err, b * N, N, a.batch * N) || (ZOH && !span_ok(a.err, c0 * N, (int64_t)nch * N, a.dim * N)))
    return;
  const uint64_t keep = policy_keep();
  if (tid == 0) {
    mbar_init(&bar, 1);
    mbar_init_fence();
  }
  __syncthreads();
  if (tid == 0) {
    mbar_expect_tx(&bar, ZOH ? 2 * bytes : bytes);
    bulk_load_hint(sst, gst, bytes, &bar, keep);
    // With the hold the arithmetic after the wait is long enough to cover A's copy, and one
    // copy of the block's A rows replaces two 16-byte loads per thread: 43.1 against 45.8 us
    // per 256 x 5120 x 16 step.  With the Euler weight the per-thread loads, which overlap
    // the wait, are faster (32.4 against 35.8 us).
    if constexpr (ZOH) bulk_load_hint(sA, a.A + c0 * N, bytes, &bar, keep);
  }
  const int cl = tid / G, l = tid % G, n0 = SPL * l;
  const bool active = cl < nch;
  const int64_t d = c0 + (active ? cl : 0);
  const int64_t c = b * a.dim + d;
  const float x = L::one(a.delta, c) + (a.delta_bias ? a.delta_bias[d] : 0.f);
  const float uu = L::one(a.u, c);
  float zz = 0.f, Dd = 0.f;
  if (l == 0) {
    if (HAS_Z) zz = L::one(a.z, c);
    if (a.D) Dd = a.D[d];
  }
  float Av[SPL], Bv[SPL], Cv[SPL], hv[SPL];
  const float* Ar = a.A + d * N + n0;
#pragma unroll
  for (int k = 0; k < SPL; k += 4) {
    const bool okn = n0 + k < N;
    if constexpr (!ZOH) {
      const float4 a4 = okn ? __ldg(reinterpret_cast<const float4*>(Ar + k)) : make_float4(0.f, 0.f, 0.f, 0.f);
      Av[k] = a4.x; Av[k + 1] = a4.y; Av[k + 2] = a4.z; Av[k + 3] = a4.w;
    }
    if (BF) {
      uint2 b2 = make_uint2(0, 0), c2 = make_uint2(0, 0);
      if (okn) {
        b2 = __ldg(reinterpret_cast<const uint2*>(static_cast<const unsigned short*>(a.B) + b * N + n0 + k));
        c2 = __ldg(reinterpret_cast<const uint2*>(static_cast<const unsigned short*>(a.C) + b * N + n0 + k));
      }
      Bv[k] = bf16_lo(b2.x); Bv[k + 1] = bf16_hi(b2.x); Bv[k + 2] = bf16_lo(b2.y); Bv[k + 3] = bf16_hi(b2.y);
      Cv[k] = bf16_lo(c2.x); Cv[k + 1] = bf16_hi(c2.x); Cv[k + 2] = bf16_lo(c2.y); Cv[k + 3] = bf16_hi(c2.y);
    } else {
      float4 b4 = make_float4(0.f, 0.f, 0.f, 0.f), c4 = b4;
      if (okn) {
        b4 = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(a.B) + b * N + n0 + k));
        c4 = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(a.C) + b * N + n0 + k));
      }
      Bv[k] = b4.x; Bv[k + 1] = b4.y; Bv[k + 2] = b4.z; Bv[k + 3] = b4.w;
      Cv[k] = c4.x; Cv[k + 1] = c4.y; Cv[k + 2] = c4.z; Cv[k + 3] = c4.w;
    }
  }
  // Every thread waits for the state's copy itself.  A thread whose wait gave up writes
  // nothing (neither its y nor its states); the block agrees at its last barrier, and the
  // state goes back to memory only if every wait succeeded.
  const bool ok = mbar_wait(&bar, 0, a.err);
  float* st = sst + cl * N + n0;
#pragma unroll
  for (int k = 0; k < SPL; k += 4) {
    const float4 h4 = (active && n0 + k < N) ? *reinterpret_cast<const float4*>(st + k) : make_float4(0.f, 0.f, 0.f, 0.f);
    hv[k] = h4.x; hv[k + 1] = h4.y; hv[k + 2] = h4.z; hv[k + 3] = h4.w;
    if constexpr (ZOH) {
      const float4 a4 = (active && n0 + k < N) ? *reinterpret_cast<const float4*>(sA + cl * N + n0 + k)
                                               : make_float4(0.f, 0.f, 0.f, 0.f);
      Av[k] = a4.x; Av[k + 1] = a4.y; Av[k + 2] = a4.z; Av[k + 3] = a4.w;
    }
  }
  const float dt = a.softplus ? softplus(x) : x;
  const float du = dt * uu;
  const f2 dtp = pk(dt, dt), dup = pk(du, du), upp = pk(uu, uu), l2e = pk(kLog2e, kLog2e);
  f2 acc = pk(0.f, 0.f);
#pragma unroll
  for (int q = 0; q < NP; ++q) {
    const f2 hq = pk(hv[2 * q], hv[2 * q + 1]);
    const f2 Aq = pk(Av[2 * q], Av[2 * q + 1]);
    const f2 arg = mul2(dtp, mul2(l2e, Aq));
    const f2 e = ex2x2(arg);
    f2 hn;
    if constexpr (ZOH) {
      const f2 iA = pk(Av[2 * q] != 0.f ? 1.f / Av[2 * q] : 0.f, Av[2 * q + 1] != 0.f ? 1.f / Av[2 * q + 1] : 0.f);
      hn = fma2(e, hq, mul2(hold2(arg, e, dtp, iA), mul2(upp, pk(Bv[2 * q], Bv[2 * q + 1]))));
    } else {
      hn = fma2(e, hq, mul2(dup, pk(Bv[2 * q], Bv[2 * q + 1])));
    }
    hv[2 * q] = lo(hn);
    hv[2 * q + 1] = hi(hn);
    acc = fma2(pk(Cv[2 * q], Cv[2 * q + 1]), hn, acc);
  }
  float y = lo(acc) + hi(acc);
  if (active && ok) {
#pragma unroll
    for (int k = 0; k < SPL; k += 4)
      if (n0 + k < N) *reinterpret_cast<float4*>(st + k) = make_float4(hv[k], hv[k + 1], hv[k + 2], hv[k + 3]);
  }
  if (G > 1) {
    const int lane = threadIdx.x & 31;
    const unsigned gmask = ((1u << G) - 1u) << (lane & ~(G - 1));
#pragma unroll
    for (int off = G / 2; off > 0; off >>= 1) y += __shfl_xor_sync(gmask, y, off);
  }
  // y sums the partial readouts of a channel's lanes: written only if every lane of the warp saw its data.
  const bool warp_ok = __all_sync(0xffffffffu, ok);
  if (active && l == 0 && warp_ok) {
    float yv = fmaf(Dd, uu, y);
    if (HAS_Z) yv *= silu(zz);
    a.y[c] = yv;
  }
  fence_async_smem();
  const bool all_ok = __syncthreads_and(ok);
  if (tid == 0) {
    if (all_ok) {
      bulk_store_hint(gst, sst, bytes, keep);
      bulk_commit();
      bulk_wait_read<0>();   // the source tile has been read: the block may exit while the write completes
    } else {
      mbar_wait(&bar, 0, nullptr);   // the copy may still be in flight: wait (bounded) before exiting
    }
  }
}

template <int NT, bool BF, bool Z>
static void go_decode(const DecodeArgs& a, int rev, cudaStream_t s) {
  constexpr int G = NT < kDecodeSpl ? 1 : NT / kDecodeSpl;
  const int64_t threads = a.dim * G;
  const dim3 g2((unsigned)((threads + kDecodeThreads - 1) / kDecodeThreads), (unsigned)a.batch);
  if constexpr (NT >= kDecodeSpl) {
    if (a.vec) {   // bulk copies of the state need 16-byte rows (N % 4 == 0) and 16-byte alignment
      if (a.zoh) decode_bulk_kernel<NT, BF, Z, true><<<g2, kDecodeThreads, 0, s>>>(a, rev);
      else decode_bulk_kernel<NT, BF, Z, false><<<g2, kDecodeThreads, 0, s>>>(a, rev);
      return;
    }
  }
  if (a.zoh) decode_kernel<NT, BF, Z, true><<<g2, kDecodeThreads, 0, s>>>(a, rev);
  else decode_kernel<NT, BF, Z, false><<<g2, kDecodeThreads, 0, s>>>(a, rev);
}

int launch_decode(const DecodeArgs& a, bool bf16, bool has_z, int reverse, cudaStream_t s) {
  SSK_DISPATCH_NT(a.dstate, {
    if (bf16) {
      if (has_z) go_decode<NT, true, true>(a, reverse, s);
      else go_decode<NT, true, false>(a, reverse, s);
    } else {
      if (has_z) go_decode<NT, false, true>(a, reverse, s);
      else go_decode<NT, false, false>(a, reverse, s);
    }
  });
  return 0;
}

}  // namespace ssk
