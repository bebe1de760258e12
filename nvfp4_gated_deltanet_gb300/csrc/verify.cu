// Commit of a verify pass: each accepted row's snapshot (the state after its
// last accepted token) is copied into the row's slot. The accepted counts are
// read on the device, so the commit can sit in a CUDA graph right after the
// acceptance decision.
#include "common.cuh"

namespace gdn {

namespace {

__global__ void __launch_bounds__(256) verify_commit_kernel(VerifyCommitArgs a) {
  const int b = blockIdx.y;
  const int slot = a.slot_ids[b];
  if (slot < 0 || slot >= a.num_slots) return;  // padding (bad ids were flagged by the verify pass)
  const int acc = a.accepted[b];
  if (acc <= 0) return;                         // nothing accepted: the slot keeps its state
  if (acc > a.r) {
    if (blockIdx.x == 0 && threadIdx.x == 0) flag_status(a.status, GDN_E_RANGE);
    return;
  }
  const size_t snap = (size_t)b * a.r + (acc - 1);
  const uint4 *ss = reinterpret_cast<const uint4 *>(static_cast<const char *>(a.snap_ssm) + snap * a.ssm_bytes);
  uint4 *sd = reinterpret_cast<uint4 *>(static_cast<char *>(a.ssm_state) + (size_t)slot * a.ssm_bytes);
  const uint4 *cs = reinterpret_cast<const uint4 *>(reinterpret_cast<const char *>(a.snap_conv) + snap * a.conv_bytes);
  uint4 *cd = reinterpret_cast<uint4 *>(reinterpret_cast<char *>(a.conv_state) + (size_t)slot * a.conv_bytes);
  const size_t nss = a.ssm_bytes / 16, ncs = a.conv_bytes / 16;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < nss; i += (size_t)gridDim.x * blockDim.x)
    sd[i] = ss[i];
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < ncs; i += (size_t)gridDim.x * blockDim.x)
    cd[i] = cs[i];
}

}  // namespace

cudaError_t launch_verify_commit(const VerifyCommitArgs &a, cudaStream_t stream) {
  if (a.B <= 0) return cudaSuccess;
  if (a.ssm_bytes % 16 || a.conv_bytes % 16) return cudaErrorInvalidValue;
  const size_t per_row = a.ssm_bytes / 16;
  int gx = (int)((per_row + 256 * 8 - 1) / (256 * 8));
  if (gx < 1) gx = 1;
  if (gx > 1024) gx = 1024;
  verify_commit_kernel<<<dim3(gx, a.B), 256, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace gdn
