// Host-side launchers shared between the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/mx.h"

namespace mx {

// Set the thread's last-error message; returns `code`.
int set_error(int code, const char* fmt, ...);

// Device properties of the current device (cached per device).
struct DeviceInfo {
  int device;  // ordinal of the current device
  int sm_count;
  int cc_major, cc_minor;
  size_t max_smem_optin;
  size_t smem_per_sm;              // shared memory of one SM
  size_t smem_reserved_per_block;  // shared memory the system reserves for each CTA
};
int current_device_info(DeviceInfo* out);

// Grid size for a grid-stride loop over `items` with `per_block` threads a block.
inline int blocks_for(long long items, int per_block) {
  long long g = (items + per_block - 1) / per_block;
  if (g > 65535LL * 8) g = 65535LL * 8;
  return g < 1 ? 1 : static_cast<int>(g);
}

// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) for `func` on the current
// device only when `bytes` exceeds what an earlier call set there (`cache`:
// one slot per device ordinal, owned by the caller's translation unit).
int raise_smem_limit(const void* func, int bytes, const DeviceInfo& di, int* cache);

// cuTensorMapEncodeTiled through the runtime's driver entry point.
int encode_tensor_map_2d(CUtensorMap* map, const void* base, CUtensorMapDataType dtype,
                         uint64_t dim0, uint64_t dim1, uint64_t stride1_bytes, uint32_t box0,
                         uint32_t box1, CUtensorMapSwizzle swizzle);

// ---- quantize / dequant (quant.cu)
// x [M, K] bf16 -> q [M, ldq] (columns K..Kout zero), codes [M, ldc] (blocks past
// K get pad_code); optional sf atoms [ceil(M/128), Kout/128, 512].  When
// `pdl_trigger` the kernel lets a programmatic dependent launch start at once.
// `M_out` (>= M, default M) rows are written; rows M..M_out-1 quantize zeros.
// `zero` / `nzero`: ints the kernel also sets to 0 (split-K arrival counters).
cudaError_t launch_quant_act(const void* x, int M, int K, int Kout, uint8_t* q, int ldq,
                             uint8_t* codes, int ldc, uint8_t pad_code, uint8_t* sf,
                             bool pdl_trigger, cudaStream_t stream, int M_out = -1,
                             int* zero = nullptr, int nzero = 0);
cudaError_t launch_dequant(const uint8_t* bytes, const uint8_t* codes, int fmt, int scale_mode,
                           int N, int K, void* out, cudaStream_t stream);

// ---- pack (pack.cu)
cudaError_t launch_pack_check_codes(const uint8_t* codes, int E, int rows, int KB, bool check_fold,
                                    unsigned int* status, cudaStream_t stream);
cudaError_t launch_pack_e4m3(const uint8_t* bytes, const uint8_t* codes, int E, int N, int K,
                             int Kp, int codes_rows, bool block_out, uint8_t* wq,
                             uint8_t* codes_out, uint8_t* sf, cudaStream_t stream);
// Activation scale atoms [ceil(M/128), Kp/128, 512] from row-major codes [M, K/32]
// (127 past M, 128 past K), the layout the GEMM's tensor-memory copy reads.
cudaError_t launch_act_sf_atoms(const uint8_t* codes, int M, int K, int Kp, uint8_t* sf, cudaStream_t stream);
cudaError_t launch_from_dequant(const void* w, const uint8_t* codes, int block_scale, int N, int K, uint8_t* out,
                                unsigned long long* mismatches, cudaStream_t stream);
cudaError_t launch_pack_e2m1(const uint8_t* bytes, const uint8_t* codes, int E, int N, int K,
                             int Kp, int codes_rows, bool gate_up, uint8_t* wq, uint8_t* codes_out,
                             uint8_t* sf, unsigned long long* negz, cudaStream_t stream);

// ---- decode GEMV (gemv.cu)
struct GemvArgs {
  const mx_packed_weight* w;
  const void* x;         // bf16 [M, K]
  const uint8_t* xq;     // [M, Kp] e4m3 (unfused path)
  const uint8_t* xcodes; // [M, Kp/32] (unfused path)
  const void* bias;      // bf16 [N] or NULL
  void* out;             // bf16 [M, N]
  int M;
  bool fused;
  bool pdl;              // launched right after the quant kernel with PDL
  int force_splits;      // 0 = heuristic
};
int launch_gemv(const GemvArgs& a, cudaStream_t stream);
unsigned int take_error_flags_gemv();
int gemv_splits(int N, int Kp, int M, int force_splits);

// ---- tensor-core decode GEMV (gemv_tc.cu): quantizes x itself, no workspace
struct TcGemvArgs {
  const mx_packed_weight* w;
  const void* x;     // bf16 [M, K]
  const void* bias;  // bf16 [N] or NULL
  void* out;         // bf16 [M, N]
  int M;             // 1..32
  const uint8_t* xq;      // pre-quantized activation [M, K] e4m3 (x unused), or NULL
  const uint8_t* xcodes;  // its codes [M, K/32]
  int force_splits;  // 0 = heuristic
  int force_ring;    // 0 = default weight ring depth
  int force_bulk;    // 1 = bulk-copy reduction at every M
  int force_cap;     // 0 = heuristic, else at most this many CTAs per SM
  int force_recv;    // 0 = heuristic, 1 = receive buffer over the weight ring, 2 = its own
};
int launch_gemv_tc(const TcGemvArgs& a, cudaStream_t stream);
int gemv_tc_splits(int N, int Kp, int sms, int force);
unsigned int take_error_flags_gemv_tc();

// ---- block-scaled GEMM (gemm.cu)
struct GemmArgs {
  const mx_packed_weight* w;
  const uint8_t* xq;    // [xq_rows, xq_cols] e4m3, row stride xq_ld bytes; rows and columns
                        // past the extent read as zeros (TMA fill)
  const uint8_t* sfa;   // [roundup(M,128)/128, Kp/128, 512] activation scale atoms
  const void* bias;     // bf16 [N] or NULL
  void* out;            // bf16 [M, N]
  int M;
  int xq_rows, xq_cols, xq_ld;  // 0: the workspace layout [roundup(M,128), Kp]
  void* part;           // room for split-K partial sums (up to gemm_part_bytes), or null: no split
  size_t part_bytes;
};
int launch_gemm(const GemmArgs& a, cudaStream_t stream);
// K ranges the GEMM splits each tile into on a device of `sms` SMs with `room`
// bytes for partial sums, and the bytes the unconstrained split takes (0: none)
int gemm_ksplit(int M, int N, int Kp, int sms, size_t room);
size_t gemm_part_bytes(int M, int N, int Kp, int sms);
unsigned int take_error_flags_gemm();

// ---- routing + MoE (moe.cu)
cudaError_t launch_route(const int32_t* ids, int T, int topk, int E, int32_t* counts,
                         int32_t* offsets, int32_t* pairs, int32_t* active, int32_t* n_active,
                         int* dev_status, cudaStream_t stream, void* zero_out = nullptr, int zero_N = 0,
                         int32_t* pass_off = nullptr, int pw = 0);
struct MoeLaunch {
  const void* x;               // bf16 [T, K] (x_per_pair = 0) or [T * topk, K] (x_per_pair = 1)
  int T, topk;
  const mx_packed_weight* w;
  const int32_t *offsets, *pairs, *active, *n_active;  // routing (mx_route_experts)
  int x_per_pair;
  int lo;                      // 1: bf16 activation as MXFP8 hi + lo pieces (A16); 0: hi only (MXFP8)
  int out_mode;                // 0: out bf16 [pairs, N]; 1: out bf16 [pairs, N/2] = silu(gate) * up; 2: out_f32
  void* out;
  void* out_f32;               // f32 [pairs, N]
  void* act;                   // activation pieces, moe_act_bytes(T * topk, Kp, E) bytes, 256-byte aligned
  size_t act_bytes;
  int wide_pass;               // pairs a wide pass (moe_wide_pass), 0: narrow passes
  const int32_t* ids;          // topk ids [T * topk] (wide passes)
  const int32_t* pass_off;     // the routing's pass offsets [E + 1] for wide_pass (wide passes)
  int no_pdl;                  // 1: launch without programmatic dependent launch
  const int32_t* inv;          // [T * topk] sorted position of each pair (-1: invalid id), or null
  void* part;                  // split-K partial sums (moe_part_bytes), or null: no split
  size_t part_bytes;
  int32_t* split_slot;         // split K: one int the GEMM writes its K-range count to (the finish reads it)
  int route_in_act;            // 1 (moe_route_in_act): the activation kernel routes ids itself and writes:
  struct {
    int32_t *offsets, *pairs, *active, *n_active;  // the routing, as mx_route_experts lays it out
    int* dev_status;           // MX_OK / MX_ERR_EXPERT_ID, or null
    void* zero_out;            // bf16 [P, zero_N] rows of invalid ids set to zero, or null
    int zero_N;
  } route;
};
size_t moe_act_bytes(long long P, int Kp, int E);
// f32 partial sums of the split-K narrow passes for P pairs of N outputs (0: never split)
size_t moe_part_bytes(long long P, int N);
// Routing for any number of pairs: route_kernel up to one chunk of pairs (inv
// untouched, returns 0), the three-kernel many-CTA routing above (scratch of
// route_scratch_bytes; fills inv, the sorted position of each pair, when given).
int route_many_writes_inv(long long P);
size_t route_scratch_bytes(long long P, int E);
cudaError_t launch_route_many(const int32_t* ids, int T, int topk, int E, int32_t* counts, int32_t* offsets,
                              int32_t* pairs, int32_t* active, int32_t* n_active, int* dev_status,
                              cudaStream_t stream, void* zero_out, int zero_N, int32_t* pass_off, int pw,
                              void* scratch, int32_t* inv);
int moe_wide_pass(long long P, int E, int lo);
// 1 when the activation kernel routes P pairs itself (at most 64 pairs, narrow passes)
int moe_route_in_act(long long P, int E, int lo);
int launch_moe(const MoeLaunch& a, cudaStream_t stream);
unsigned int take_error_flags_moe();
unsigned int take_error_flags_selftest();
cudaError_t launch_combine(const float* y2, const int32_t* ids, const float* wts, int T, int topk, int E, int H,
                           void* out, cudaStream_t stream);

}  // namespace mx
