// C ABI of the library (include/mx.h): argument checks, workspace carving and
// dispatch to the kernels.  No call allocates memory; only mx_pack_weights and
// mx_check_device_errors synchronise.

#include <cudaTypedefs.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "mx_common.cuh"
#include "mx_internal.h"

namespace mx {

namespace {
thread_local char g_msg[512] = {0};

constexpr size_t kAlign = 256;
constexpr int kFusedQuantMaxM = 8;  // quantize x inside the GEMV up to this many tokens

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
int padded_k(int K) { return (K + 127) / 128 * 128; }

struct DevCache {
  bool valid;
  DeviceInfo info;
};
DevCache g_dev[64];
std::mutex g_dev_mu;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

int check_device() {
  DeviceInfo di;
  const int rc = current_device_info(&di);
  if (rc != MX_OK) return rc;
  if (di.cc_major != 10 || di.cc_minor != 3)
    return set_error(MX_ERR_UNSUPPORTED, "device compute capability %d.%d is not sm_103", di.cc_major,
                     di.cc_minor);
  return MX_OK;
}

int cuda_fail(cudaError_t e, const char* what) {
  return set_error(MX_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Packed-buffer regions: [header 256 B][bytes][codes][sf]
struct PackRegions {
  size_t bytes_off, codes_off, sf_off, total;
};

PackRegions pack_regions(int fmt, int E, int N, int K) {
  PackRegions r;
  const int Kp = padded_k(K);
  // E2M1: 128-row tiles, so N rounds up to a multiple of 128
  const size_t nbytes = fmt == MX_FMT_E4M3 ? static_cast<size_t>(E) * N * Kp
                                           : static_cast<size_t>(E) * ((N + 127) / 128) * 128 * (Kp / 2);
  const size_t ncodes = static_cast<size_t>(E) * N * (Kp / 32);  // row mode is the larger
  const size_t nsf = static_cast<size_t>(E) * ((N + 127) / 128) * (Kp / 128) * 512;
  r.bytes_off = kAlign;
  r.codes_off = r.bytes_off + align_up(nbytes, kAlign);
  r.sf_off = r.codes_off + align_up(ncodes, kAlign);
  r.total = r.sf_off + align_up(nsf, kAlign);
  return r;
}

struct LinearWs {
  size_t xq_off, codes_off, part_off, total;  // part_off: the bytes the call needs
};

// SM count the GEMM's K split is sized for: the current device's, else the
// GB300's 152 (a host without a device still gets a size).
int gemm_sizing_sms() {
  int dev = 0, v = 0;
  if (cudaGetDevice(&dev) == cudaSuccess && cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
      v > 0)
    return v;
  cudaGetLastError();
  return 152;
}

// Workspace of the cluster GEMV (M <= 32) and of the GEMM (M > 32): quantized
// activation [Mp, Kp] and its codes / scale atoms (required), then room for
// the GEMM's K-range partial sums (when its tiles leave SMs idle; a smaller
// workspace gets fewer ranges).  The tensor-core GEMV (M <= 32, the default)
// quantizes in shared memory and needs none.
LinearWs linear_ws(int M, int N, int Kp) {
  LinearWs r;
  const size_t Mp = M <= MX_GEMV_MAX_M ? static_cast<size_t>(M) : (static_cast<size_t>(M) + 127) / 128 * 128;
  r.xq_off = 0;
  r.codes_off = align_up(Mp * Kp, kAlign);
  r.part_off = r.codes_off + align_up(Mp * (Kp / 32), kAlign);
  const size_t part = M > MX_GEMV_MAX_M ? gemm_part_bytes(M, N, Kp, gemm_sizing_sms()) : 0;
  r.total = r.part_off + align_up(part, kAlign);
  return r;
}

struct MoeWs {
  size_t counts, offsets, pairs, inv, active, n_active, status, pass_off, route_tmp, act, act_bytes, part,
      part_bytes, total;
};

// Routing outputs, then the activation pieces of the T * topk pairs for K
// values padded to Kp (Kp = 0: routing only), then the split-K partial sums
// for N outputs a pair.
MoeWs moe_ws(int T, int topk, int E, int N, int Kp) {
  MoeWs r;
  const size_t P = static_cast<size_t>(T) * topk;
  size_t o = 0;
  r.counts = o;   o += align_up(4 * static_cast<size_t>(E), 16);
  r.offsets = o;  o += align_up(4 * (static_cast<size_t>(E) + 1), 16);
  r.pairs = o;    o += align_up(4 * (P ? P : 1), 16);
  r.inv = o;      o += align_up(4 * (P ? P : 1), 16);
  r.active = o;   o += align_up(4 * static_cast<size_t>(E), 16);
  r.n_active = o; o += 16;
  r.status = o;   o += 16;
  r.pass_off = o; o += align_up(4 * (static_cast<size_t>(E) + 1), 16);
  r.route_tmp = o; o += align_up(route_scratch_bytes(static_cast<long long>(P), E), 16);
  r.act = align_up(o, 256);
  r.act_bytes = Kp > 0 ? moe_act_bytes(static_cast<long long>(P), Kp, E) : 0;
  r.part = align_up(r.act + r.act_bytes, 256);
  r.part_bytes = Kp > 0 ? moe_part_bytes(static_cast<long long>(P), N) : 0;
  r.total = r.part + r.part_bytes;
  return r;
}

}  // namespace

int set_error(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return code;
}

int current_device_info(DeviceInfo* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return set_error(MX_ERR_UNSUPPORTED, "device ordinal %d", dev);
  std::lock_guard<std::mutex> lock(g_dev_mu);
  if (!g_dev[dev].valid) {
    DeviceInfo di = {};
    int v = 0;
    if ((e = cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_fail(e, "device attribute");
    di.sm_count = v;
    di.device = dev;
    cudaDeviceGetAttribute(&di.cc_major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&di.cc_minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    di.max_smem_optin = static_cast<size_t>(v);
    cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    di.smem_per_sm = static_cast<size_t>(v);
    v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrReservedSharedMemoryPerBlock, dev);
    di.smem_reserved_per_block = static_cast<size_t>(v);
    g_dev[dev].info = di;
    g_dev[dev].valid = true;
  }
  *out = g_dev[dev].info;
  return MX_OK;
}

int raise_smem_limit(const void* func, int bytes, const DeviceInfo& di, int* cache) {
  int* slot = cache + di.device;
  if (__atomic_load_n(slot, __ATOMIC_ACQUIRE) >= bytes) return MX_OK;
  const cudaError_t e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return cuda_fail(e, "shared memory attribute");
  int cur = __atomic_load_n(slot, __ATOMIC_ACQUIRE);
  while (cur < bytes && !__atomic_compare_exchange_n(slot, &cur, bytes, false, __ATOMIC_ACQ_REL, __ATOMIC_ACQUIRE)) {
  }
  return MX_OK;
}

int encode_tensor_map_2d(CUtensorMap* map, const void* base, CUtensorMapDataType dtype,
                         uint64_t dim0, uint64_t dim1, uint64_t stride1_bytes, uint32_t box0,
                         uint32_t box1, CUtensorMapSwizzle swizzle) {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!g_encode) return set_error(MX_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
  // A map depends only on these parameters, never on the memory's contents:
  // the last 64 distinct ones are kept (a decode loop re-encodes the same
  // weight maps every call).
  struct Key {
    const void* base;
    uint64_t dim0, dim1, stride1;
    uint32_t box0, box1;
    int dtype, swizzle;
  };
  static Key keys[64];
  static CUtensorMap maps[64];
  static bool used[64];
  static std::mutex mu;
  const Key k = {base, dim0, dim1, stride1_bytes, box0, box1, static_cast<int>(dtype), static_cast<int>(swizzle)};
  const size_t slot = ((reinterpret_cast<uintptr_t>(base) >> 8) ^ (dim0 * 31u) ^ (dim1 * 131u) ^ box1 ^
                       (static_cast<uint64_t>(dtype) << 5)) & 63u;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (used[slot] && std::memcmp(&keys[slot], &k, sizeof(Key)) == 0) {
      *map = maps[slot];
      return MX_OK;
    }
  }
  const cuuint64_t dims[2] = {dim0, dim1};
  const cuuint64_t strides[1] = {stride1_bytes};
  const cuuint32_t box[2] = {box0, box1};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = g_encode(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return set_error(MX_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
  std::lock_guard<std::mutex> lock(mu);
  keys[slot] = k;
  maps[slot] = *map;
  used[slot] = true;
  return MX_OK;
}

}  // namespace mx

using namespace mx;

extern "C" {

const char* mx_last_error(void) { return g_msg; }

int mx_check_device_errors(void) {
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
  const unsigned int flags =
      take_error_flags_gemv() | take_error_flags_gemm() | take_error_flags_gemv_tc() | take_error_flags_moe() |
      take_error_flags_selftest();
  if (flags & 0x80000000u) return set_error(MX_ERR_CUDA, "could not read the device error flags");
  if (flags & 1u) return set_error(MX_ERR_TIMEOUT, "a bounded wait inside a kernel timed out");
  return MX_OK;
}

size_t mx_pack_size(int fmt, int E, int N, int K) {
  if ((fmt != MX_FMT_E4M3 && fmt != MX_FMT_E2M1) || E < 1 || N < 1 || K < 32 || K % 32) return 0;
  return pack_regions(fmt, E, N, K).total;
}

int mx_pack_weights(const uint8_t* bytes, const uint8_t* codes, int fmt, int E, int N, int K,
                    int codes_rows, unsigned flags, void* dst, size_t dst_bytes,
                    mx_packed_weight* out, void* stream_) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  if (fmt != MX_FMT_E4M3 && fmt != MX_FMT_E2M1) return set_error(MX_ERR_ARG, "unknown format %d", fmt);
  if (!bytes || !codes || !dst || !out) return set_error(MX_ERR_ARG, "NULL pointer");
  if (E < 1 || N < 1 || K < 32 || K % 32)
    return set_error(MX_ERR_SHAPE, "E=%d N=%d K=%d: need E, N >= 1 and K a positive multiple of 32", E, N, K);
  const bool rows_given = codes_rows == N;
  const bool blocks_given = !rows_given && N % 32 == 0 && codes_rows == N / 32;
  if (!rows_given && !blocks_given)
    return set_error(MX_ERR_SHAPE, "codes_rows=%d must be N=%d or N/32", codes_rows, N);
  if (flags & ~(MX_PACK_FOLD | MX_PACK_REQUIRE_BLOCK | MX_PACK_GATE_UP))
    return set_error(MX_ERR_ARG, "unknown pack flags");
  const bool gate_up = (flags & MX_PACK_GATE_UP) != 0;
  if (gate_up && fmt != MX_FMT_E2M1) return set_error(MX_ERR_ARG, "MX_PACK_GATE_UP applies to E2M1 experts");
  if (gate_up && N % 16 != 0) return set_error(MX_ERR_SHAPE, "MX_PACK_GATE_UP needs N = 2 I a multiple of 16");
  if (!aligned16(bytes) || (reinterpret_cast<uintptr_t>(dst) % kAlign))
    return set_error(MX_ERR_ALIGN, "weight bytes need 16-byte and dst 256-byte alignment");
  const PackRegions R = pack_regions(fmt, E, N, K);
  if (dst_bytes < R.total) return set_error(MX_ERR_SHAPE, "dst holds %zu bytes, needs %zu", dst_bytes, R.total);
  int rc = check_device();
  if (rc != MX_OK) return rc;

  uint8_t* base = static_cast<uint8_t*>(dst);
  unsigned int* status = reinterpret_cast<unsigned int*>(base);
  unsigned long long* negz = reinterpret_cast<unsigned long long*>(base + 8);
  const int Kp = padded_k(K);
  const int KB = K / 32;
  const bool want_fold = fmt == MX_FMT_E4M3 && rows_given && N % 32 == 0 &&
                         (flags & (MX_PACK_FOLD | MX_PACK_REQUIRE_BLOCK));
  cudaError_t e = cudaMemsetAsync(base, 0, kAlign, stream);
  if (e != cudaSuccess) return cuda_fail(e, "pack: memset");
  if ((e = launch_pack_check_codes(codes, E, codes_rows, KB, want_fold, status, stream)) != cudaSuccess)
    return cuda_fail(e, "pack: check codes");
  unsigned int st = 0;
  if ((e = cudaMemcpyAsync(&st, status, sizeof(st), cudaMemcpyDeviceToHost, stream)) != cudaSuccess)
    return cuda_fail(e, "pack: read status");
  if ((e = cudaStreamSynchronize(stream)) != cudaSuccess) return cuda_fail(e, "pack: synchronize");
  if (st & 1u) return set_error(MX_ERR_SCALE, "an E8M0 weight code is 255 (NaN)");

  mx_packed_weight w = {};
  w.fmt = fmt;
  w.E = E;
  w.N = N;
  w.K = K;
  w.Kp = Kp;
  w.bytes = base + R.bytes_off;
  w.codes = base + R.codes_off;
  w.sf = base + R.sf_off;
  if (fmt == MX_FMT_E4M3) {
    bool block;
    if (blocks_given) {
      block = true;
    } else if (want_fold && !(st & 2u)) {
      block = true;
    } else {
      if (flags & MX_PACK_REQUIRE_BLOCK)
        return set_error(MX_ERR_NOT_BLOCK32, "row scales [%d, %d] are not 32 x 32 blocks", N, KB);
      block = false;
    }
    w.scale_mode = block ? MX_SCALE_BLOCK32X32 : MX_SCALE_ROW1X32;
    if ((e = launch_pack_e4m3(bytes, codes, E, N, K, Kp, codes_rows, block, w.bytes, w.codes, w.sf, stream)) !=
        cudaSuccess)
      return cuda_fail(e, "pack e4m3");
  } else {
    w.scale_mode = MX_SCALE_ROW1X32;
    w.layout = gate_up ? MX_LAYOUT_GATE_UP : MX_LAYOUT_PLAIN;
    e = launch_pack_e2m1(bytes, codes, E, N, K, Kp, codes_rows, gate_up, w.bytes, w.codes, w.sf, negz, stream);
    if (e != cudaSuccess) return cuda_fail(e, "pack e2m1");
  }
  unsigned long long nz = 0;
  if ((e = cudaMemcpyAsync(&nz, negz, sizeof(nz), cudaMemcpyDeviceToHost, stream)) != cudaSuccess)
    return cuda_fail(e, "pack: read -0 count");
  if ((e = cudaStreamSynchronize(stream)) != cudaSuccess) return cuda_fail(e, "pack: synchronize");
  w.neg_zero_count = static_cast<int64_t>(nz);
  *out = w;
  return MX_OK;
}

int mx_quantize_act(const void* x, int M, int K, uint8_t* q, uint8_t* codes, void* stream) {
  if (M < 0 || K < 32 || K % 32) return set_error(MX_ERR_SHAPE, "M=%d K=%d: K must be a positive multiple of 32", M, K);
  if (M == 0) return MX_OK;
  if (!x || !q || !codes) return set_error(MX_ERR_ARG, "NULL pointer");
  if (!aligned16(x) || !aligned16(q)) return set_error(MX_ERR_ALIGN, "x and q need 16-byte alignment");
  int rc = check_device();
  if (rc != MX_OK) return rc;
  cudaError_t e = launch_quant_act(x, M, K, K, q, K, codes, K / 32, 128, nullptr, false,
                                   static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MX_OK : cuda_fail(e, "quantize launch");
}

int mx_e4m3_from_dequant(const void* w, const uint8_t* codes, int scale_mode, int N, int K, uint8_t* out,
                         void* scratch, int64_t* mismatches, void* stream_) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  if (mismatches) *mismatches = 0;
  if (scale_mode != MX_SCALE_BLOCK32X32 && scale_mode != MX_SCALE_ROW1X32)
    return set_error(MX_ERR_ARG, "unknown scale mode %d", scale_mode);
  if (N < 0 || K < 32 || K % 32) return set_error(MX_ERR_SHAPE, "N=%d K=%d", N, K);
  if (scale_mode == MX_SCALE_BLOCK32X32 && N % 32) return set_error(MX_ERR_SHAPE, "32x32 blocks need N %% 32 == 0");
  if (N == 0) return MX_OK;
  if (!w || !codes || !out || !scratch) return set_error(MX_ERR_ARG, "NULL pointer");
  if (!aligned16(w) || !aligned16(out) || (reinterpret_cast<uintptr_t>(scratch) & 7u))
    return set_error(MX_ERR_ALIGN, "w and out need 16-byte, scratch 8-byte alignment");
  int rc = check_device();
  if (rc != MX_OK) return rc;
  unsigned long long* cnt = static_cast<unsigned long long*>(scratch);
  cudaError_t e = cudaMemsetAsync(cnt, 0, sizeof(*cnt), stream);
  if (e != cudaSuccess) return cuda_fail(e, "from_dequant: memset");
  if ((e = launch_from_dequant(w, codes, scale_mode == MX_SCALE_BLOCK32X32 ? 1 : 0, N, K, out, cnt, stream)) !=
      cudaSuccess)
    return cuda_fail(e, "from_dequant launch");
  unsigned long long host = 0;
  if ((e = cudaMemcpyAsync(&host, cnt, sizeof(host), cudaMemcpyDeviceToHost, stream)) != cudaSuccess)
    return cuda_fail(e, "from_dequant: read count");
  if ((e = cudaStreamSynchronize(stream)) != cudaSuccess) return cuda_fail(e, "from_dequant: synchronize");
  if (mismatches) *mismatches = static_cast<int64_t>(host);
  if (host) return set_error(MX_ERR_INEXACT, "%llu of %lld values are not e4m3 x scale", host,
                             static_cast<long long>(N) * K);
  return MX_OK;
}

int mx_dequant(const uint8_t* bytes, const uint8_t* codes, int fmt, int scale_mode, int N, int K,
               void* out, void* stream) {
  if (fmt != MX_FMT_E4M3 && fmt != MX_FMT_E2M1) return set_error(MX_ERR_ARG, "unknown format %d", fmt);
  if (scale_mode != MX_SCALE_BLOCK32X32 && scale_mode != MX_SCALE_ROW1X32)
    return set_error(MX_ERR_ARG, "unknown scale mode %d", scale_mode);
  if (N < 0 || K < 32 || K % 32) return set_error(MX_ERR_SHAPE, "N=%d K=%d", N, K);
  if (scale_mode == MX_SCALE_BLOCK32X32 && N % 32) return set_error(MX_ERR_SHAPE, "32x32 blocks need N %% 32 == 0");
  if (N == 0) return MX_OK;
  if (!bytes || !codes || !out) return set_error(MX_ERR_ARG, "NULL pointer");
  if (!aligned16(bytes) || !aligned16(out)) return set_error(MX_ERR_ALIGN, "bytes and out need 16-byte alignment");
  int rc = check_device();
  if (rc != MX_OK) return rc;
  cudaError_t e = launch_dequant(bytes, codes, fmt, scale_mode, N, K, out, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MX_OK : cuda_fail(e, "dequant launch");
}

size_t mxfp8_linear_workspace_size(int M, const mx_packed_weight* w) {
  if (!w || M <= 0) return 0;
  return linear_ws(M, w->N, w->Kp).total;
}

int mxfp8_linear(const void* x, int M, const mx_packed_weight* w, const void* bias, void* out,
                 unsigned flags, void* workspace, size_t workspace_bytes, void* stream_) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  if (!w) return set_error(MX_ERR_ARG, "NULL weight");
  if (w->fmt != MX_FMT_E4M3 || w->E != 1) return set_error(MX_ERR_ARG, "mxfp8_linear needs a dense E4M3 weight");
  if (M < 0) return set_error(MX_ERR_SHAPE, "M=%d", M);
  if (M == 0) return MX_OK;
  if (!x || !out) return set_error(MX_ERR_ARG, "NULL pointer");
  if (!aligned16(x) || !aligned16(out) || (bias && !aligned16(bias)))
    return set_error(MX_ERR_ALIGN, "x, out and bias need 16-byte alignment");
  int rc = check_device();
  if (rc != MX_OK) return rc;
  // tuning overrides of the cluster GEMV (not part of the documented flags):
  // bits 8..11 force its split count, bit 12 forces its fused quantizer;
  // bits 16..18 force the tensor-core GEMV's weight ring depth, bit 23 its
  // bulk-copy reduction at every M, bits 24..26 its CTAs per SM, bits 27..28
  // its receive-buffer placement
  const int force_splits = static_cast<int>((flags >> 8) & 0xfu);
  const bool force_fuse = (flags & (1u << 12)) != 0;
  const bool no_fuse = (flags & MX_LINEAR_NO_FUSED_QUANT) != 0;
  const bool legacy = (flags & MX_LINEAR_CLUSTER_GEMV) != 0;
  const int Kp = w->Kp;
  const LinearWs L = linear_ws(M, w->N, Kp);

  auto run_chunk = [&](const void* xc, int Mc, void* oc) -> int {
    GemvArgs a = {};
    a.w = w;
    a.x = xc;
    a.bias = bias;
    a.out = oc;
    a.M = Mc;
    a.force_splits = force_splits;
    if ((Mc <= kFusedQuantMaxM || force_fuse) && !no_fuse) {
      a.fused = true;
      return launch_gemv(a, stream);
    }
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    a.xq = ws + L.xq_off;
    a.xcodes = ws + L.codes_off;
    cudaError_t e = launch_quant_act(xc, Mc, w->K, Kp, ws + L.xq_off, Kp, ws + L.codes_off, Kp / 32, 127,
                                     nullptr, true, stream);
    if (e != cudaSuccess) return cuda_fail(e, "quantize launch");
    a.fused = false;
    a.pdl = true;
    return launch_gemv(a, stream);
  };

  if (M <= MX_GEMV_MAX_M && !legacy) {
    TcGemvArgs g = {};
    g.w = w;
    g.x = x;
    g.bias = bias;
    g.out = out;
    g.M = M;
    g.force_splits = force_splits;
    g.force_ring = static_cast<int>((flags >> 16) & 0x7u);      // tuning: weight ring depth
    g.force_bulk = (flags >> 23) & 1u;                          // tuning: bulk-copy reduction
    g.force_cap = static_cast<int>((flags >> 24) & 0x7u);       // tuning: CTAs per SM
    g.force_recv = static_cast<int>((flags >> 27) & 0x3u);      // tuning: receive-buffer placement
    if (no_fuse) {
      // the fused quant switched off: x quantized by its own launch (the same
      // block rule, so the same bits) into the workspace, which the GEMV reads
      // after its dependency wait
      if (!workspace || workspace_bytes < L.total)
        return set_error(MX_ERR_WORKSPACE, "workspace of %zu bytes, needs %zu", workspace_bytes, L.total);
      if (!aligned16(workspace)) return set_error(MX_ERR_ALIGN, "workspace needs 16-byte alignment");
      uint8_t* ws = static_cast<uint8_t*>(workspace);
      cudaError_t e = launch_quant_act(x, M, w->K, w->K, ws + L.xq_off, w->K, ws + L.codes_off, w->K / 32, 128,
                                       nullptr, true, stream);
      if (e != cudaSuccess) return cuda_fail(e, "quantize launch");
      g.x = nullptr;
      g.xq = ws + L.xq_off;
      g.xcodes = ws + L.codes_off;
    }
    return launch_gemv_tc(g, stream);
  }
  const bool needs_ws = (M > kFusedQuantMaxM && !force_fuse) || no_fuse || M > MX_GEMV_MAX_M;
  if (needs_ws && (!workspace || workspace_bytes < L.part_off))
    return set_error(MX_ERR_WORKSPACE, "workspace of %zu bytes, needs %zu", workspace_bytes, L.part_off);
  if (needs_ws && !aligned16(workspace)) return set_error(MX_ERR_ALIGN, "workspace needs 16-byte alignment");
  const bool force_gemv = (flags & (1u << 13)) != 0;  // tuning: chunked GEMV for M > 32
  if (M > MX_GEMV_MAX_M && !force_gemv) {
    // block-scaled GEMM: quantize into [Mp, Kp] + activation scale atoms, then tcgen05
    const int Mp = (M + 127) / 128 * 128;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    cudaError_t e = launch_quant_act(x, M, w->K, Kp, ws + L.xq_off, Kp, nullptr, 0, 127, ws + L.codes_off,
                                     true, stream, Mp);
    if (e != cudaSuccess) return cuda_fail(e, "quantize launch");
    GemmArgs g = {};
    g.w = w;
    g.xq = ws + L.xq_off;
    g.sfa = ws + L.codes_off;
    g.bias = bias;
    g.out = out;
    g.M = M;
    if (workspace_bytes > L.part_off) {
      g.part = ws + L.part_off;
      g.part_bytes = workspace_bytes - L.part_off;
    }
    return launch_gemm(g, stream);
  }
  const size_t xrow = static_cast<size_t>(w->K) * 2, orow = static_cast<size_t>(w->N) * 2;
  for (int m0 = 0; m0 < M; m0 += MX_GEMV_MAX_M) {
    const int Mc = (M - m0) < MX_GEMV_MAX_M ? (M - m0) : MX_GEMV_MAX_M;
    rc = run_chunk(static_cast<const uint8_t*>(x) + m0 * xrow, Mc, static_cast<uint8_t*>(out) + m0 * orow);
    if (rc != MX_OK) return rc;
  }
  return MX_OK;
}

// the activation's scale atoms, then the GEMM's K-range partial sums (if any)
static size_t q_atoms_bytes(int M, const mx_packed_weight* w) {
  return align_up(static_cast<size_t>((M + 127) / 128) * (w->Kp / 128) * 512, kAlign);
}

size_t mxfp8_linear_q_workspace_size(int M, const mx_packed_weight* w) {
  if (!w || M <= MX_GEMV_MAX_M) return 0;
  return q_atoms_bytes(M, w) + align_up(gemm_part_bytes(M, w->N, w->Kp, gemm_sizing_sms()), kAlign);
}

int mxfp8_linear_q(const uint8_t* xq, const uint8_t* xcodes, int M, const mx_packed_weight* w, const void* bias,
                   void* out, unsigned flags, void* workspace, size_t workspace_bytes, void* stream_) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  if (!w) return set_error(MX_ERR_ARG, "NULL weight");
  if (w->fmt != MX_FMT_E4M3 || w->E != 1) return set_error(MX_ERR_ARG, "mxfp8_linear_q needs a dense E4M3 weight");
  if (flags != 0) return set_error(MX_ERR_ARG, "mxfp8_linear_q takes no flags");
  if (M < 0) return set_error(MX_ERR_SHAPE, "M=%d", M);
  if (M == 0) return MX_OK;
  if (!xq || !xcodes || !out) return set_error(MX_ERR_ARG, "NULL pointer");
  if (!aligned16(xq) || !aligned16(out) || (bias && !aligned16(bias)))
    return set_error(MX_ERR_ALIGN, "xq, out and bias need 16-byte alignment");
  int rc = check_device();
  if (rc != MX_OK) return rc;
  if (M <= MX_GEMV_MAX_M) {
    TcGemvArgs g = {};
    g.w = w;
    g.xq = xq;
    g.xcodes = xcodes;
    g.bias = bias;
    g.out = out;
    g.M = M;
    return launch_gemv_tc(g, stream);
  }
  const size_t need = q_atoms_bytes(M, w);  // the partial sums take what room is left
  if (!workspace || workspace_bytes < need)
    return set_error(MX_ERR_WORKSPACE, "workspace of %zu bytes, needs %zu", workspace_bytes, need);
  if (!aligned16(workspace)) return set_error(MX_ERR_ALIGN, "workspace needs 16-byte alignment");
  uint8_t* sfa = static_cast<uint8_t*>(workspace);
  cudaError_t e = launch_act_sf_atoms(xcodes, M, w->K, w->Kp, sfa, stream);
  if (e != cudaSuccess) return cuda_fail(e, "scale atoms launch");
  GemmArgs g = {};
  g.w = w;
  g.xq = xq;          // [M, K]: rows past M and columns past K read as zeros
  g.xq_rows = M;
  g.xq_cols = w->K;
  g.xq_ld = w->K;
  g.sfa = sfa;
  g.bias = bias;
  g.out = out;
  g.M = M;
  if (workspace_bytes > need) {
    g.part = sfa + need;
    g.part_bytes = workspace_bytes - need;
  }
  return launch_gemm(g, stream);
}

int mx_route_experts(const int32_t* topk_ids, int T, int topk, int E, int32_t* counts,
                     int32_t* offsets, int32_t* pairs, int32_t* active, int32_t* n_active,
                     int* dev_status, void* stream) {
  if (T < 0 || topk < 1 || E < 1) return set_error(MX_ERR_SHAPE, "T=%d topk=%d E=%d", T, topk, E);
  if (E > MX_MAX_EXPERTS) return set_error(MX_ERR_UNSUPPORTED, "E=%d exceeds %d", E, MX_MAX_EXPERTS);
  if ((T > 0 && !topk_ids) || !counts || !offsets || !pairs || !active || !n_active)
    return set_error(MX_ERR_ARG, "NULL pointer");
  int rc = check_device();
  if (rc != MX_OK) return rc;
  cudaError_t e = launch_route(topk_ids, T, topk, E, counts, offsets, pairs, active, n_active, dev_status,
                               static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MX_OK : cuda_fail(e, "route launch");
}

size_t mxfp4_moe_workspace_size(int T, int topk, int E, int N, int K) {
  if (T < 0 || topk < 1 || E < 1 || N < 1 || K < 32 || K % 32) return 0;
  return moe_ws(T, topk, E, N, padded_k(K)).total;
}

// (internal) the routed expert GEMM with bf16 activations (lo = 1: hi and lo
// MXFP8 pieces) or MXFP8-quantized activations (lo = 0: hi alone)
static int moe_linear_impl(int lo, const char* name, const void* x, const int32_t* topk_ids, int T, int topk,
                           const mx_packed_weight* w, void* out, void* workspace, size_t workspace_bytes,
                           int* dev_status, void* stream_) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  if (!w) return set_error(MX_ERR_ARG, "NULL weight");
  if (w->fmt != MX_FMT_E2M1) return set_error(MX_ERR_ARG, "%s needs an E2M1 weight", name);
  if (T < 0 || topk < 1) return set_error(MX_ERR_SHAPE, "T=%d topk=%d", T, topk);
  if (w->E > MX_MAX_EXPERTS) return set_error(MX_ERR_UNSUPPORTED, "E=%d exceeds %d", w->E, MX_MAX_EXPERTS);
  if (T == 0) return MX_OK;
  if (!x || !topk_ids || !out || !workspace) return set_error(MX_ERR_ARG, "NULL pointer");
  if (!aligned16(x) || !aligned16(out) || !aligned16(workspace))
    return set_error(MX_ERR_ALIGN, "x, out and workspace need 16-byte alignment");
  const MoeWs R = moe_ws(T, topk, w->E, w->N, w->Kp);
  if (workspace_bytes < R.total) return set_error(MX_ERR_WORKSPACE, "workspace of %zu bytes, needs %zu", workspace_bytes, R.total);
  int rc = check_device();
  if (rc != MX_OK) return rc;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int32_t* counts = reinterpret_cast<int32_t*>(ws + R.counts);
  int32_t* offsets = reinterpret_cast<int32_t*>(ws + R.offsets);
  int32_t* pairs = reinterpret_cast<int32_t*>(ws + R.pairs);
  int32_t* active = reinterpret_cast<int32_t*>(ws + R.active);
  int32_t* n_active = reinterpret_cast<int32_t*>(ws + R.n_active);
  int* st = dev_status ? dev_status : reinterpret_cast<int*>(ws + R.status);
  // routing (with pass offsets when the experts average enough pairs for wide
  // passes), and zero rows for the pairs whose id is not a valid expert; at
  // decode sizes the activation kernel routes
  const long long P = static_cast<long long>(T) * topk;
  const int pw = moe_wide_pass(P, w->E, lo);
  int32_t* pass_off = reinterpret_cast<int32_t*>(ws + R.pass_off);
  int32_t* inv = reinterpret_cast<int32_t*>(ws + R.inv);
  MoeLaunch a = {};
  a.route_in_act = moe_route_in_act(P, w->E, lo);
  if (a.route_in_act) {
    a.route.offsets = offsets;
    a.route.pairs = pairs;
    a.route.active = active;
    a.route.n_active = n_active;
    a.route.dev_status = st;
    a.route.zero_out = out;
    a.route.zero_N = w->N;
  } else {
    cudaError_t e = launch_route_many(topk_ids, T, topk, w->E, counts, offsets, pairs, active, n_active, st, stream,
                                      out, w->N, pw ? pass_off : nullptr, pw, ws + R.route_tmp, inv);
    if (e != cudaSuccess) return cuda_fail(e, "route launch");
  }
  a.x = x;
  a.T = T;
  a.topk = topk;
  a.w = w;
  a.offsets = offsets;
  a.pairs = pairs;
  a.active = active;
  a.n_active = n_active;
  a.lo = lo;
  a.out_mode = 0;
  a.out = out;
  a.act = ws + R.act;
  a.act_bytes = R.act_bytes;
  a.part = ws + R.part;
  a.part_bytes = R.part_bytes;
  a.split_slot = n_active + 1;  // the n_active slot is 16 bytes
  a.wide_pass = pw;
  a.ids = topk_ids;
  a.pass_off = pass_off;
  a.inv = route_many_writes_inv(static_cast<long long>(T) * topk) ? inv : nullptr;
  return launch_moe(a, stream);
}

int mxfp4_moe_linear(const void* x, const int32_t* topk_ids, int T, int topk, const mx_packed_weight* w,
                     void* out, void* workspace, size_t workspace_bytes, int* dev_status, void* stream) {
  return moe_linear_impl(1, "mxfp4_moe_linear", x, topk_ids, T, topk, w, out, workspace, workspace_bytes,
                         dev_status, stream);
}

int mxfp4_moe_linear_w4a8(const void* x, const int32_t* topk_ids, int T, int topk, const mx_packed_weight* w,
                          void* out, void* workspace, size_t workspace_bytes, int* dev_status, void* stream) {
  return moe_linear_impl(0, "mxfp4_moe_linear_w4a8", x, topk_ids, T, topk, w, out, workspace, workspace_bytes,
                         dev_status, stream);
}

// (internal: static inside the extern "C" block)
struct ExpertWs {
  MoeWs route;
  size_t act, y2, total;
};

static ExpertWs expert_ws(int T, int topk, int E, int K, int I, int H) {
  ExpertWs r;
  // the activation pieces serve both projections in turn: sized for the longer K
  const int Kp = padded_k(K) > padded_k(I) ? padded_k(K) : padded_k(I);
  // the partial sums serve both projections in turn: sized for the wider N
  r.route = moe_ws(T, topk, E, 2 * I > H ? 2 * I : H, Kp);
  const size_t P = static_cast<size_t>(T) * topk;
  r.act = align_up(r.route.total, 256);
  r.y2 = align_up(r.act + P * static_cast<size_t>(I) * 2, 256);
  r.total = r.y2 + P * static_cast<size_t>(H) * 4;
  return r;
}

size_t mxfp4_moe_expert_workspace_size(int T, int topk, int E, int K, int I, int H) {
  if (T < 0 || topk < 1 || E < 1 || K < 32 || K % 32 || I < 32 || I % 32 || H < 1) return 0;
  return expert_ws(T, topk, E, K, I, H).total;
}

int mxfp4_moe_expert(const void* x, const int32_t* topk_ids, const float* topk_weights, int T, int topk,
                     const mx_packed_weight* w13, const mx_packed_weight* w2, void* out, void* workspace,
                     size_t workspace_bytes, int* dev_status, void* stream_) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  if (!w13 || !w2) return set_error(MX_ERR_ARG, "NULL weight");
  if (w13->fmt != MX_FMT_E2M1 || w2->fmt != MX_FMT_E2M1)
    return set_error(MX_ERR_ARG, "mxfp4_moe_expert needs E2M1 weights");
  if (w13->layout != MX_LAYOUT_GATE_UP)
    return set_error(MX_ERR_ARG, "w13 must be packed with MX_PACK_GATE_UP");
  if (w2->layout != MX_LAYOUT_PLAIN) return set_error(MX_ERR_ARG, "w2 must be packed without MX_PACK_GATE_UP");
  const int I = w13->N / 2, H = w2->N, E = w13->E;
  if (w2->E != E || w2->K != I)
    return set_error(MX_ERR_SHAPE, "w2 [E=%d, H=%d, K=%d] does not fit w13 [E=%d, 2I=%d]", w2->E, H, w2->K, E,
                     w13->N);
  if (H % 4 != 0) return set_error(MX_ERR_SHAPE, "H=%d must be a multiple of 4", H);
  if (T < 0 || topk < 1) return set_error(MX_ERR_SHAPE, "T=%d topk=%d", T, topk);
  if (E > MX_MAX_EXPERTS) return set_error(MX_ERR_UNSUPPORTED, "E=%d exceeds %d", E, MX_MAX_EXPERTS);
  if (T == 0) return MX_OK;
  if (!x || !topk_ids || !topk_weights || !out || !workspace) return set_error(MX_ERR_ARG, "NULL pointer");
  if (!aligned16(x) || !aligned16(out) || !aligned16(workspace))
    return set_error(MX_ERR_ALIGN, "x, out and workspace need 16-byte alignment");
  const ExpertWs R = expert_ws(T, topk, E, w13->K, I, H);
  if (workspace_bytes < R.total)
    return set_error(MX_ERR_WORKSPACE, "workspace of %zu bytes, needs %zu", workspace_bytes, R.total);
  int rc = check_device();
  if (rc != MX_OK) return rc;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int32_t* counts = reinterpret_cast<int32_t*>(ws + R.route.counts);
  int32_t* offsets = reinterpret_cast<int32_t*>(ws + R.route.offsets);
  int32_t* pairs = reinterpret_cast<int32_t*>(ws + R.route.pairs);
  int32_t* active = reinterpret_cast<int32_t*>(ws + R.route.active);
  int32_t* n_active = reinterpret_cast<int32_t*>(ws + R.route.n_active);
  int* st = dev_status ? dev_status : reinterpret_cast<int*>(ws + R.route.status);
  const long long P = static_cast<long long>(T) * topk;
  const int pw = moe_wide_pass(P, E, 1);
  int32_t* pass_off = reinterpret_cast<int32_t*>(ws + R.route.pass_off);
  int32_t* inv = reinterpret_cast<int32_t*>(ws + R.route.inv);
  cudaError_t e = cudaSuccess;
  MoeLaunch a = {};
  // at decode sizes the gate / up activation kernel routes (the down
  // projection then reads its routing)
  a.route_in_act = moe_route_in_act(P, E, 1);
  if (a.route_in_act) {
    a.route.offsets = offsets;
    a.route.pairs = pairs;
    a.route.active = active;
    a.route.n_active = n_active;
    a.route.dev_status = st;
  } else {
    e = launch_route_many(topk_ids, T, topk, E, counts, offsets, pairs, active, n_active, st, stream, nullptr, 0,
                          pw ? pass_off : nullptr, pw, ws + R.route.route_tmp, inv);
    if (e != cudaSuccess) return cuda_fail(e, "route launch");
  }
  a.wide_pass = pw;
  a.ids = topk_ids;
  a.pass_off = pass_off;
  a.inv = route_many_writes_inv(static_cast<long long>(T) * topk) ? inv : nullptr;
  a.T = T;
  a.topk = topk;
  a.lo = 1;
  a.act = ws + R.route.act;
  a.act_bytes = R.route.act_bytes;
  a.part = ws + R.route.part;
  a.part_bytes = R.route.part_bytes;
  a.split_slot = n_active + 1;  // the n_active slot is 16 bytes
  a.offsets = offsets;
  a.pairs = pairs;
  a.active = active;
  a.n_active = n_active;
  // gate / up with SiLU-and-mul fused: act [T * topk, I] bf16
  a.x = x;
  a.w = w13;
  a.x_per_pair = 0;
  a.out_mode = 1;
  a.out = ws + R.act;
  if ((rc = launch_moe(a, stream)) != MX_OK) return rc;
  a.route_in_act = 0;
  // down projection: one activation row a pair, f32 [T * topk, H].  Launched
  // without programmatic dependent launch: letting its kernels start while the
  // gate/up GEMM drains cost ~6 us a call at E=64 I=2048 H=4096 T=64 (GB300)
  a.no_pdl = 1;
  a.x = ws + R.act;
  a.w = w2;
  a.x_per_pair = 1;
  a.out_mode = 2;
  a.out = nullptr;
  a.out_f32 = ws + R.y2;
  if ((rc = launch_moe(a, stream)) != MX_OK) return rc;
  if ((e = launch_combine(reinterpret_cast<const float*>(ws + R.y2), topk_ids, topk_weights, T, topk, E, H, out,
                          stream)) != cudaSuccess)
    return cuda_fail(e, "combine launch");
  return MX_OK;
}

}  // extern "C"
