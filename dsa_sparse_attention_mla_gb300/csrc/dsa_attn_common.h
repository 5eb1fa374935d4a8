// dsa_attn_common.h - host-side pieces shared by the attention kernels' translation units:
// the Q tensor map, the split-token workspace layout and the per-call merge-flag epoch.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include "dsa_host.h"

namespace dsa {

constexpr int kAttnHeads = 64;

// 3-D tiled map over q [T][64][dk] bf16 (strides from the call), box 64 x 64 x 1, 128-byte
// swizzle: one box is a 64-column chunk of all heads of one token, in the K-major SW128 layout
// the MMA reads.
dsa_status_t encode_q_tensor_map(const dsa_attn_args_t* a, int dk, CUtensorMap* out);

// Per-workspace call counter (never 0): the merge flags of a call carry its value, so flags left
// by an earlier call, even one that stopped on a timeout, never match.
int next_attn_epoch(const void* workspace);

// Workspace of the split-token merge, per persistent CTA b: partial o [b][64 * 256] fp32,
// running values [b][4][64] fp32 (max, sum, and the 8-bit-operand kernel's two output-half
// maxima) and eight publish flags [b][8] int32; then the work-balanced split:
// valid-entry counts of 32 unit slices per CTA and the G + 1 range bounds, int64.
size_t attn_ws_bytes(int sm_count);
struct AttnWorkspace {
  float* o;
  float* ml;
  int* flags;
  int64_t* split;
};
AttnWorkspace attn_ws_layout(void* workspace, int sm_count);

// Work split of a keys-as-M launch over (token, 128-entry window) units: one persistent CTA per
// SM with at least 4 units each and at most 17 CTAs per token; for long batches, a split by
// work whose range bounds two small pre-pass kernels compute on `stream` (into ws.split).
struct UnitSplit {
  int G;                  // CTAs
  int NT;                 // 128-entry windows per token
  int64_t U;              // units (T * NT)
  const int64_t* bounds;  // G + 1 range bounds on the device, or null for equal unit counts
  int gap;                // fewest units a balanced range may hold
};
dsa_status_t plan_unit_split(const dsa_attn_args_t* a, const DeviceInfo& dev, const AttnWorkspace& ws,
                             cudaStream_t stream, UnitSplit* out);

// One-time set-up, per device, of every attention kernel (the dynamic shared-memory limit is a
// per-device attribute of each kernel). Every attention entry point runs it before its first
// launch on a device; it does nothing on later calls.
dsa_status_t prepare_attn_kernels(int device);
// Sets the attributes of the keys-as-M kernels on the current device (part of the above).
cudaError_t k128_set_attributes();

// Sets the attribute of the 8-bit-operand kernel on the current device (part of the above).
cudaError_t f8_set_attributes();

// The 256+0 latent geometry: packed FP8 rows run the 8-bit-operand kernel (dsa_attn_f8.cu),
// bf16 rows the keys-as-M bf16 kernel (dsa_attn_k128.cu).
dsa_status_t launch_attn_f8(const dsa_attn_args_t* a, const DeviceInfo& dev, cudaStream_t stream);

// The 512+64 control geometry over packed FP8 rows: keys-as-M with 8-bit operands, 32 heads per
// work unit (dsa_attn_ctl.cu).
cudaError_t ctl_set_attributes();
dsa_status_t launch_attn_ctl(const dsa_attn_args_t* a, const DeviceInfo& dev, cudaStream_t stream);

// Keys-as-M kernel for the 256+0 latent geometry (dsa_attn_k128.cu); routes packed FP8 rows
// to launch_attn_f8.
dsa_status_t launch_attn_k128(const dsa_attn_args_t* a, const DeviceInfo& dev, cudaStream_t stream);

}  // namespace dsa
