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
// (max, sum) [b][2][64] fp32 and eight publish flags [b][8] int32; then the work-balanced split:
// valid-entry counts of 32 unit slices per CTA and the G + 1 range bounds, int64.
size_t attn_ws_bytes(int sm_count);
struct AttnWorkspace {
  float* o;
  float* ml;
  int* flags;
  int64_t* split;
};
AttnWorkspace attn_ws_layout(void* workspace, int sm_count);

// One-time set-up, per device, of every attention kernel (the dynamic shared-memory limit is a
// per-device attribute of each kernel). Every attention entry point runs it before its first
// launch on a device; it does nothing on later calls.
dsa_status_t prepare_attn_kernels(int device);
// Sets the attributes of the keys-as-M kernels on the current device (part of the above).
cudaError_t k128_set_attributes();

// Keys-as-M kernel for the 256+0 latent geometry (dsa_attn_k128.cu).
dsa_status_t launch_attn_k128(const dsa_attn_args_t* a, const DeviceInfo& dev, cudaStream_t stream);

}  // namespace dsa
