// Device helpers shared by the MX kernels: PTX wrappers for mbarriers, TMA,
// ldmatrix, warp MMAs, format conversions, bounded waits and PDL.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/mx.h"

#define MX_DEV __device__ __forceinline__

namespace mx {

// Device error flags of this translation unit (bit 0: a bounded wait timed
// out).  Each unit with bounded waits exports a host reader (take_error_flags_*)
// that mx_check_device_errors() calls.
static __device__ unsigned int g_error_flags = 0;

// Host side: read and clear this unit's flags (the device must be idle).
static inline unsigned int take_tu_error_flags() {
  unsigned int f = 0, z = 0;
  if (cudaMemcpyFromSymbol(&f, g_error_flags, sizeof(f)) != cudaSuccess) return 0x80000000u;
  if (cudaMemcpyToSymbol(g_error_flags, &z, sizeof(z)) != cudaSuccess) return 0x80000000u;
  return f;
}

// Bounded waits give up after this many nanoseconds of %globaltimer.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s

MX_DEV uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

MX_DEV unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

MX_DEV void flag_timeout() { atomicOr(&g_error_flags, 1u); }

// ------------------------------------------------------------------ mbarrier

MX_DEV void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

MX_DEV void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

MX_DEV void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

MX_DEV void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

MX_DEV bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// try_wait with cluster-scope acquire: the waiting thread sees every write
// that peers of the cluster completed on this barrier (st.async complete_tx).
MX_DEV bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase with the given parity to complete.  Gives up after
// limit_ns of %globaltimer, sets the device timeout flag and returns false.
MX_DEV bool mbar_wait_for(uint64_t* bar, uint32_t parity, unsigned long long limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 0 && globaltimer() - t0 > limit_ns) {
      flag_timeout();
      return false;
    }
  }
}

// mbar_wait_for with the library's limit, kWaitLimitNs.
MX_DEV bool mbar_wait(uint64_t* bar, uint32_t parity) { return mbar_wait_for(bar, parity, kWaitLimitNs); }

// mbar_wait with cluster-scope acquire (bounded the same way).
MX_DEV bool mbar_wait_cluster(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if ((i & 255u) == 0 && globaltimer() - t0 > kWaitLimitNs) {
      flag_timeout();
      return false;
    }
  }
}

// --------------------------------------------------------------------- TMA

MX_DEV void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

// 2D tiled load of one box into shared memory, completing on `bar`.
MX_DEV void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y,
                        uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
      "l"(map), "r"(smem_u32(bar)), "r"(x), "r"(y), "l"(policy)
      : "memory");
}

MX_DEV uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

MX_DEV uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

MX_DEV void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------- PDL (griddepcontrol)

MX_DEV void pdl_wait_prior_grid() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
MX_DEV void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------------ cluster

MX_DEV uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

MX_DEV void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

// The two halves of a cluster barrier, for threads that reach them at
// different points of divergent code (no .aligned).  Every thread of every CTA
// of the cluster arrives once per phase before any of them may pass the wait.
MX_DEV void cluster_arrive_release() { asm volatile("barrier.cluster.arrive.release;" ::: "memory"); }
MX_DEV void cluster_wait_acquire() { asm volatile("barrier.cluster.wait.acquire;" ::: "memory"); }

// Shared-memory address of the same variable in CTA `rank` of the cluster.
MX_DEV uint32_t map_shared_rank(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

// Four floats into the shared memory of a CTA of the cluster (addresses from
// map_shared_rank, 16-byte aligned); their 16 bytes complete on that CTA's
// mbarrier `bar` (complete_tx), which orders them for its waiting threads.
MX_DEV void st_async_v4_f32(uint32_t addr, float a, float b, float c, float d, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                   addr),
               "f"(a), "f"(b), "f"(c), "f"(d), "r"(bar)
               : "memory");
}

// Bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned) from
// this CTA's shared memory into the shared memory of a CTA of the cluster
// (dst and bar from map_shared_rank); the bytes complete on that CTA's mbarrier.
MX_DEV void bulk_copy_to_peer(uint32_t dst, uint32_t src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   dst),
               "r"(src), "r"(bytes), "r"(bar)
               : "memory");
}
MX_DEV void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Waits until the committed bulk copies have read their sources.
MX_DEV void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// Barrier over the `count` threads (a multiple of 32) that use barrier `id` (1..15).
MX_DEV void named_barrier(uint32_t id, uint32_t count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Store to the shared memory of another CTA of the cluster (address from map_shared_rank).
MX_DEV void st_shared_cluster_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// Not volatile: independent loads may be issued back to back.  Ordering against
// the peers' writes comes from the cluster barrier that precedes every use.
MX_DEV float ld_shared_cluster_f32(uint32_t addr) {
  float v;
  asm("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr));
  return v;
}

// ---------------------------------------------------------- loads / ldmatrix

MX_DEV uint4 ld_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

MX_DEV void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

MX_DEV void ldsm_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];"
               : "=r"(r0), "=r"(r1)
               : "r"(addr));
}

// ------------------------------------------------------------------ warp MMA

// D = A(16x32 e4m3, row) * B(32x8 e4m3, col), fp32 accumulate from zero.
MX_DEV void mma_e4m3_16832(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.0f));
}

// C += A(16x16 bf16, row) * B(16x8 bf16, col), fp32 accumulate.
MX_DEV void mma_bf16_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                           uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ------------------------------------------------------------ conversions

// E8M0 code -> 2^(c - 127) as f32; code 0 -> 2^-127 (subnormal); 255 -> NaN.
MX_DEV float e8m0_to_f32(uint32_t c) {
  if (c == 0u) return __uint_as_float(0x00400000u);
  if (c == 255u) return __uint_as_float(0x7fc00000u);
  return __uint_as_float(c << 23);
}

// Two f32 -> packed e4m3x2 (lo = first element at the lower address), RNE,
// finite values clamped to +-448 (never reached by the quantizer), NaN kept.
MX_DEV uint32_t f32x2_to_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Packed e4m3x2 -> two f16 (exact).
MX_DEV __half2 e4m3x2_to_f16x2(uint16_t v) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(v));
  return *reinterpret_cast<__half2*>(&r);
}

// Packed e2m1x2 (one byte, low nibble = first element) -> two f16 (exact).
MX_DEV __half2 e2m1x2_to_f16x2(uint32_t byte) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}"
      : "=r"(r)
      : "r"(byte));
  return *reinterpret_cast<__half2*>(&r);
}

// --------------------------------------------------------- MXFP8 quantizer
//
// rocm_native, _quant_mxfp8_tile: per 32-element block, amax = max(max|x|, 2^-126),
// code = clamp(ceil(log2(amax / 448)) + 127, 0, 254), q = e4m3(x * 2^(127 - code)).
// Four consecutive lanes (aligned) hold one block, 8 elements each.  The code is
// taken from amax's exponent and mantissa bits: with amax = 1.f * 2^ex (amax is a
// normal f32 because it is at least 2^-126), ceil(log2(amax / 448)) equals
// ex - 8 when 1.f <= 1.75 and ex - 7 otherwise, since 448 = 1.75 * 2^8.

struct QuantBlock8 {
  uint32_t lo, hi;  // 8 e4m3 bytes, element 0 in the lowest byte of lo
  uint32_t code;    // E8M0 code of the block
};

MX_DEV uint32_t mx_block_code(float amax) {
  const uint32_t bits = __float_as_uint(fmaxf(amax, 1.17549435e-38f));
  const int ex = static_cast<int>(bits >> 23) - 127;
  const int e = ex - 8 + ((bits & 0x7fffffu) > 0x600000u ? 1 : 0);
  const int c = e + 127;
  return static_cast<uint32_t>(c < 0 ? 0 : (c > 254 ? 254 : c));
}

MX_DEV void bf16x8_to_f32(const uint4& u, float (&v)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

// One whole MX block in one thread: u[0..3] hold the block's 32 bf16 elements
// in order (8 per uint4, element 0 in the low half of u[0].x).  Same rule and
// same bits as mx_quant_bf16x8, without shuffles: out[0..1] receive the 32
// e4m3 bytes (element 0 in the lowest byte of out[0].x), the return value is
// the E8M0 code (255 for a block with NaN or inf, bytes 0x7F).
MX_DEV uint32_t mx_quant_bf16x32(const uint4 (&u)[4], uint4 (&out)[2]) {
  uint32_t m2 = 0u;
#pragma unroll
  for (int q = 0; q < 4; ++q)
    m2 = __vmaxu2(m2, __vmaxu2(__vmaxu2(u[q].x & 0x7fff7fffu, u[q].y & 0x7fff7fffu),
                               __vmaxu2(u[q].z & 0x7fff7fffu, u[q].w & 0x7fff7fffu)));
  const uint32_t m = max(m2 & 0xffffu, m2 >> 16);
  if (m >= 0x7f80u) {  // NaN or inf in the block
    out[0] = out[1] = make_uint4(0x7f7f7f7fu, 0x7f7f7f7fu, 0x7f7f7f7fu, 0x7f7f7f7fu);
    return 255u;
  }
  const uint32_t code = mx_block_code(__uint_as_float(m << 16));
  const uint32_t ef = 254u - code;
  const float rescale = ef ? __uint_as_float(ef << 23) : __uint_as_float(0x00400000u);
  uint32_t w[8];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint32_t in[4] = {u[q].x, u[q].y, u[q].z, u[q].w};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t p0 = f32x2_to_e4m3x2(__uint_as_float(in[2 * h] << 16) * rescale,
                                          __uint_as_float(in[2 * h] & 0xffff0000u) * rescale);
      const uint32_t p1 = f32x2_to_e4m3x2(__uint_as_float(in[2 * h + 1] << 16) * rescale,
                                          __uint_as_float(in[2 * h + 1] & 0xffff0000u) * rescale);
      w[2 * q + h] = p0 | (p1 << 16);
    }
  }
  out[0] = make_uint4(w[0], w[1], w[2], w[3]);
  out[1] = make_uint4(w[4], w[5], w[6], w[7]);
  return code;
}

// u: this lane's 8 consecutive bf16 elements of the block (element 0 in the
// low half of u.x); 4 consecutive lanes hold the 32 elements of one block.
// The block maximum is taken on the bf16 bit patterns with the sign cleared:
// for finite values their unsigned order is the order of the magnitudes, inf
// is 0x7f80 and every NaN lies above it.
MX_DEV QuantBlock8 mx_quant_bf16x8(const uint4& u) {
  const uint32_t m2 = __vmaxu2(__vmaxu2(u.x & 0x7fff7fffu, u.y & 0x7fff7fffu),
                               __vmaxu2(u.z & 0x7fff7fffu, u.w & 0x7fff7fffu));
  uint32_t m = max(m2 & 0xffffu, m2 >> 16);
  m = max(m, __shfl_xor_sync(0xffffffffu, m, 1));
  m = max(m, __shfl_xor_sync(0xffffffffu, m, 2));
  QuantBlock8 r;
  if (m >= 0x7f80u) {  // NaN or inf in the block
    r.lo = r.hi = 0x7f7f7f7fu;
    r.code = 255u;
    return r;
  }
  const uint32_t code = mx_block_code(__uint_as_float(m << 16));
  // 2^(127 - code): exponent field 254 - code; 0 -> the subnormal 2^-127
  const uint32_t ef = 254u - code;
  const float rescale = ef ? __uint_as_float(ef << 23) : __uint_as_float(0x00400000u);
  float v[8];
  bf16x8_to_f32(u, v);
  const uint32_t p0 = f32x2_to_e4m3x2(v[0] * rescale, v[1] * rescale);
  const uint32_t p1 = f32x2_to_e4m3x2(v[2] * rescale, v[3] * rescale);
  const uint32_t p2 = f32x2_to_e4m3x2(v[4] * rescale, v[5] * rescale);
  const uint32_t p3 = f32x2_to_e4m3x2(v[6] * rescale, v[7] * rescale);
  r.lo = p0 | (p1 << 16);
  r.hi = p2 | (p3 << 16);
  r.code = code;
  return r;
}

}  // namespace mx
