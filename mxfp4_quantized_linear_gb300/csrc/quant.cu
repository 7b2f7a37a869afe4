// K-QUANT (per-token MXFP8 activation quantizer) and K-DEQ (MX dequant to bf16).
//
// Quantizer: rocm_native (vllm.model_executor.kernels.linear.mxfp8.rocm_native),
// _quant_mxfp8_tile.  Dequant: weights942, ocp_from_dequant (w = e4m3 value x
// 2^(code - 127)) and a16w4, dequant (fp4x2, low nibble first).
//
// Both are HBM-bound elementwise passes: each thread moves 16 bytes of bf16,
// four lanes form one 32-element MX block.

#include "mx_common.cuh"
#include "mx_internal.h"

namespace mx {

namespace {

// One thread = one whole 32-element MX block (64 bytes of bf16 in, 32 e4m3
// bytes and one code out), two blocks in flight a thread; consecutive threads
// take consecutive blocks of a row, so a warp reads 2 KB and writes 1 KB
// contiguously.  Grid-stride over the blocks of the [M_out, Kout] output
// (Kout >= K, multiple of 32); 32-bit index arithmetic (M_out * Kout / 32 <
// 2^31 is checked by the launcher).
__global__ void __launch_bounds__(256) quant_act_kernel(const __nv_bfloat16* __restrict__ x,
                                                        int M, int K, int Kout,
                                                        uint8_t* __restrict__ q, int ldq,
                                                        uint8_t* __restrict__ codes, int ldc,
                                                        uint8_t pad_code, uint8_t* __restrict__ sf,
                                                        int pdl_trigger, int M_out, int* zero,
                                                        int nzero) {
  if (pdl_trigger) {
    // launched as a programmatic dependent: let the next kernel start, but
    // touch x and the outputs only once the previous kernel is complete
    pdl_launch_dependents();
    pdl_wait_prior_grid();
  }
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < nzero; i += gridDim.x * blockDim.x) zero[i] = 0;
  const unsigned KBo = static_cast<unsigned>(Kout) >> 5, KB = static_cast<unsigned>(K) >> 5;
  const unsigned total = static_cast<unsigned>(M_out) * KBo;
  const unsigned stride = gridDim.x * blockDim.x;
  for (unsigned b0 = blockIdx.x * blockDim.x + threadIdx.x; b0 < total; b0 += 2 * stride) {
    uint4 u[2][4];
    unsigned row[2], kb[2];
    bool valid[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const unsigned b = b0 + j * stride;
      row[j] = b / KBo;
      kb[j] = b - row[j] * KBo;
      valid[j] = b < total && row[j] < static_cast<unsigned>(M) && kb[j] < KB;
#pragma unroll
      for (int c = 0; c < 4; ++c) u[j][c] = make_uint4(0u, 0u, 0u, 0u);
      if (valid[j]) {
        const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<long long>(row[j]) * K + kb[j] * 32);
#pragma unroll
        for (int c = 0; c < 4; ++c) u[j][c] = src[c];
      }
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const unsigned b = b0 + j * stride;
      if (b >= total) break;
      uint4 o[2];
      uint32_t code = mx_quant_bf16x32(u[j], o);  // zeros -> zero bytes, code 0
      // blocks past K get pad_code; rows past M are quantized zeros (code 0)
      if (!valid[j] && kb[j] >= KB) code = pad_code;
      uint4* dst = reinterpret_cast<uint4*>(q + static_cast<long long>(row[j]) * ldq + kb[j] * 32);
      dst[0] = o[0];
      dst[1] = o[1];
      const uint8_t c8 = static_cast<uint8_t>(code);
      if (codes) codes[static_cast<long long>(row[j]) * ldc + kb[j]] = c8;
      if (sf) {
        // 512-byte atom (row tile, 128-K tile): row m, block kb at (m%32)*16 + (m/32)*4 + kb%4
        const unsigned m = row[j] & 127u;
        const long long atom = static_cast<long long>(row[j] >> 7) * (KBo >> 2) + (kb[j] >> 2);
        sf[atom * 512 + (m & 31u) * 16 + (m >> 5) * 4 + (kb[j] & 3u)] = c8;
      }
    }
  }
}

// Dequant: one thread = 8 consecutive output elements of a row.
template <int kFmt>
__global__ void __launch_bounds__(256) dequant_kernel(const uint8_t* __restrict__ bytes,
                                                      const uint8_t* __restrict__ codes,
                                                      int block_scale, int N, int K,
                                                      __nv_bfloat16* __restrict__ out) {
  const int groups_per_row = K >> 3;
  const long long total = static_cast<long long>(N) * groups_per_row;
  const int KB = K >> 5;
  for (long long g = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; g < total;
       g += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int n = static_cast<int>(g / groups_per_row);
    const int k = static_cast<int>(g % groups_per_row) * 8;
    const int crow = block_scale ? (n >> 5) : n;
    const float s = e8m0_to_f32(codes[static_cast<long long>(crow) * KB + (k >> 5)]);
    float v[8];
    if (kFmt == MX_FMT_E4M3) {
      const uint2 u = *reinterpret_cast<const uint2*>(bytes + static_cast<long long>(n) * K + k);
      const uint32_t w[2] = {u.x, u.y};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const __half2 h = e4m3x2_to_f16x2(static_cast<uint16_t>(w[i >> 1] >> (16 * (i & 1))));
        const float2 f = __half22float2(h);
        v[2 * i] = f.x;
        v[2 * i + 1] = f.y;
      }
    } else {
      const uint32_t w =
          *reinterpret_cast<const uint32_t*>(bytes + static_cast<long long>(n) * (K >> 1) + (k >> 1));
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = __half22float2(e2m1x2_to_f16x2((w >> (8 * i)) & 0xffu));
        v[2 * i] = f.x;
        v[2 * i + 1] = f.y;
      }
    }
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat162 b = __floats2bfloat162_rn(v[2 * i] * s, v[2 * i + 1] * s);
      o[i] = *reinterpret_cast<const uint32_t*>(&b);
    }
    *reinterpret_cast<uint4*>(out + static_cast<long long>(n) * K + k) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// weights942, ocp_from_dequant: the e4m3 bytes behind a bf16 weight w = e4m3
// value x 2^(code - 127).  One thread = 8 consecutive elements of a row: scale
// by 2^(127 - code), round to e4m3 (nearest-even, saturating: a value beyond
// 448 fails the check below anyway), and count the values whose byte does not
// give w back (dequant rounded to bf16; -0 equals +0, a NaN never matches).
__global__ void __launch_bounds__(256) from_dequant_kernel(const __nv_bfloat16* __restrict__ w,
                                                           const uint8_t* __restrict__ codes,
                                                           int block_scale, int N, int K,
                                                           uint8_t* __restrict__ out,
                                                           unsigned long long* mismatches) {
  const int groups_per_row = K >> 3;
  const long long total = static_cast<long long>(N) * groups_per_row;
  const int KB = K >> 5;
  unsigned int bad = 0;
  for (long long g = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; g < total;
       g += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int n = static_cast<int>(g / groups_per_row);
    const int k = static_cast<int>(g % groups_per_row) * 8;
    const uint32_t c = codes[static_cast<long long>(block_scale ? (n >> 5) : n) * KB + (k >> 5)];
    const uint4 u = *reinterpret_cast<const uint4*>(w + static_cast<long long>(n) * K + k);
    const uint32_t wb[4] = {u.x, u.y, u.z, u.w};
    uint32_t o[2] = {0x7f7f7f7fu, 0x7f7f7f7fu};
    if (c == 255u) {
      bad += 8;  // a NaN scale gives nothing back
    } else {
      // 2^(127 - c) and 2^(c - 127) as f32: exponent fields 254 - c and c, 0 -> 2^-127
      const float down = (c == 254u) ? __uint_as_float(0x00400000u) : __uint_as_float((254u - c) << 23);
      const float up = (c == 0u) ? __uint_as_float(0x00400000u) : __uint_as_float(c << 23);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t lo = wb[i] & 0xffffu, hi = wb[i] >> 16;
        const uint32_t q = f32x2_to_e4m3x2(__uint_as_float(lo << 16) * down, __uint_as_float(hi << 16) * down);
        const float2 f = __half22float2(e4m3x2_to_f16x2(static_cast<uint16_t>(q)));
        const __nv_bfloat162 b = __floats2bfloat162_rn(f.x * up, f.y * up);
        const uint32_t bb = *reinterpret_cast<const uint32_t*>(&b);
        const uint32_t blo = bb & 0xffffu, bhi = bb >> 16;
        const bool ok_lo = ((blo == lo) || (((blo | lo) & 0x7fffu) == 0)) && (lo & 0x7fffu) <= 0x7f80u;
        const bool ok_hi = ((bhi == hi) || (((bhi | hi) & 0x7fffu) == 0)) && (hi & 0x7fffu) <= 0x7f80u;
        bad += (ok_lo ? 0u : 1u) + (ok_hi ? 0u : 1u);
        // bytes 2i, 2i + 1 of the 8 outputs
        const uint32_t shift = 16u * (i & 1);
        o[i >> 1] = (o[i >> 1] & ~(0xffffu << shift)) | (q << shift);
      }
    }
    *reinterpret_cast<uint2*>(out + static_cast<long long>(n) * K + k) = make_uint2(o[0], o[1]);
  }
  for (int off = 16; off > 0; off >>= 1) bad += __shfl_xor_sync(0xffffffffu, bad, off);
  if ((threadIdx.x & 31) == 0 && bad) atomicAdd(mismatches, static_cast<unsigned long long>(bad));
}

int grid_for(long long threads, int block) {
  long long g = (threads + block - 1) / block;
  DeviceInfo di;
  const int cap = (current_device_info(&di) == MX_OK) ? di.sm_count * 16 : 2048;
  if (g > cap) g = cap;
  return g < 1 ? 1 : static_cast<int>(g);
}

}  // namespace

cudaError_t launch_quant_act(const void* x, int M, int K, int Kout, uint8_t* q, int ldq,
                             uint8_t* codes, int ldc, uint8_t pad_code, uint8_t* sf,
                             bool pdl_trigger, cudaStream_t stream, int M_out, int* zero,
                             int nzero) {
  if (M_out < M) M_out = M;
  const long long blocks = static_cast<long long>(M_out) * (Kout / 32);
  if (blocks >= (1LL << 31)) return cudaErrorInvalidValue;  // the kernel indexes blocks in 32 bits
  const int block = 256;
  const int grid = grid_for((blocks + 1) / 2, block);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(block, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = pdl_trigger ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, quant_act_kernel, static_cast<const __nv_bfloat16*>(x), M, K, Kout, q, ldq,
                            codes, ldc, pad_code, sf, pdl_trigger ? 1 : 0, M_out, zero, nzero);
}

cudaError_t launch_from_dequant(const void* w, const uint8_t* codes, int block_scale, int N, int K, uint8_t* out,
                                unsigned long long* mismatches, cudaStream_t stream) {
  const long long groups = static_cast<long long>(N) * (K / 8);
  const int grid = grid_for(groups, 256);
  from_dequant_kernel<<<grid, 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(w), codes, block_scale, N, K, out,
                                                mismatches);
  return cudaGetLastError();
}

cudaError_t launch_dequant(const uint8_t* bytes, const uint8_t* codes, int fmt, int scale_mode,
                           int N, int K, void* out, cudaStream_t stream) {
  const long long groups = static_cast<long long>(N) * (K / 8);
  const int block = 256;
  const int grid = grid_for(groups, block);
  const int blk = scale_mode == MX_SCALE_BLOCK32X32 ? 1 : 0;
  if (fmt == MX_FMT_E4M3)
    dequant_kernel<MX_FMT_E4M3><<<grid, block, 0, stream>>>(bytes, codes, blk, N, K,
                                                             static_cast<__nv_bfloat16*>(out));
  else
    dequant_kernel<MX_FMT_E2M1><<<grid, block, 0, stream>>>(bytes, codes, blk, N, K,
                                                             static_cast<__nv_bfloat16*>(out));
  return cudaGetLastError();
}

}  // namespace mx
