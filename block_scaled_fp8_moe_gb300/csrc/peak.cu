// Block-scaled tensor-core rate probe: the denominator of the prefill roofline.
//
// The grouped GEMMs run tcgen05.mma kind::mxf8f6f4 (E2M1 weights x E4M3 activations, UE8M0 scales
// per 32 along K; "New Deepseek 4.1 flash recipe", post 6 "How it works" item 1). Their tensor
// utilisation is quoted against what that instruction itself sustains on this GPU, measured here:
// one CTA per SM issues back-to-back M = 128, N = 256, K = 32 MMAs into one TMEM accumulator from
// operands that stay resident in shared memory (no copies, no epilogue), so the only limit is the
// tensor pipe. The caller times the launch with CUDA events; FLOPs = 2 * 128 * 256 * 32 * iters *
// CTAs. Not part of the layer.
#include <cuda_runtime.h>

#include "common.cuh"
#include "ptx.cuh"

namespace moe {

constexpr int kProbeN = 256;
constexpr int kProbeThreads = 128;
// more than half of an SM's shared memory, so no two probe CTAs share an SM (each allocates all
// 512 TMEM columns)
constexpr int kProbeSmem = 128 * 1024;
constexpr uint64_t kProbeWaitNs = 1000000000ull;

__device__ __forceinline__ uint32_t probe_hash(uint32_t v) {
  v ^= v >> 16;
  v *= 0x7feb352du;
  v ^= v >> 15;
  v *= 0x846ca68bu;
  v ^= v >> 16;
  return v;
}

__global__ void __launch_bounds__(kProbeThreads, 1) mma_rate_probe_kernel(int iters, uint32_t* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = base;                          // 128 rows x 128 B (E2M1 in 8-bit containers)
  uint8_t* sB = sA + 128 * 128;                // 256 rows x 128 B (E4M3)
  uint8_t* sSF = sB + kProbeN * 128;           // A scale atom (512 B), then two B scale atoms
  uint64_t* done = reinterpret_cast<uint64_t*>(sSF + 3 * 512);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  const int warp = threadIdx.x >> 5;

  // operands: pseudo-random bytes (every E2M1 code is finite; E4M3 NaN codes are moved to the
  // neighbouring finite code), scales 2^0
  for (int i = threadIdx.x; i < 128 * 128 + kProbeN * 128; i += kProbeThreads) {
    uint8_t b = (uint8_t)probe_hash((uint32_t)i * 2654435761u + blockIdx.x);
    if (i >= 128 * 128 && (b & 0x7f) == 0x7f) b -= 1;
    base[i] = b;
  }
  for (int i = threadIdx.x; i < 3 * 512; i += kProbeThreads) sSF[i] = 127;
  fence_async_smem();
  if (threadIdx.x == 0) {
    mbar_init(done, 1);
    mbar_fence_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (warp == 0 && (threadIdx.x & 31) == 0) {
    const uint32_t tsfa = tmem + 256, tsfb = tsfa + 4;
    tc_cp_32x128b_warpx4(tsfa, smem_desc(smem_u32(sSF), 16, 128, 0));
    tc_cp_32x128b_warpx4(tsfb, smem_desc(smem_u32(sSF + 512), 16, 128, 0));
    tc_cp_32x128b_warpx4(tsfb + 4, smem_desc(smem_u32(sSF + 1024), 16, 128, 0));
    const uint32_t idesc0 = idesc_mxf8f6f4(5 /*E2M1*/, 0 /*E4M3*/, 128, kProbeN, 0, 0);
    const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
    for (int it = 0; it < iters; ++it) {
      const int kb = it & 3;
      const uint32_t id = idesc0 | ((uint32_t)kb << 4) | ((uint32_t)kb << 29);
      mma_mxf8f6f4(tmem, smem_desc(a0 + kb * 32, 16, 1024, 2), smem_desc(b0 + kb * 32, 16, 1024, 2), id, tsfa, tsfb,
                   it > 0 ? 1u : 0u);
    }
    tc_commit(done);
    mbar_wait(done, 0, kProbeWaitNs, nullptr, status, DEV_TIMEOUT_DRAIN);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

}  // namespace moe

using namespace moe;

extern "C" int moe_probe_mma_rate(int32_t iters, int32_t* ctas, int64_t* flops, void* ws, size_t ws_bytes,
                                  void* stream) {
  if (iters <= 0 || iters > (1 << 24) || !ctas || !flops) return MOE_ERR_INVALID_ARG;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255) || ws_bytes < 256) return MOE_ERR_WORKSPACE;
  if (ensure_smem_limit((const void*)mma_rate_probe_kernel, kProbeSmem + 1024)) return MOE_ERR_CUDA;
  const int grid = num_sms();
  *ctas = grid;
  *flops = 2LL * 128 * kProbeN * 32 * (int64_t)iters * grid;
  mma_rate_probe_kernel<<<grid, kProbeThreads, kProbeSmem + 1024, static_cast<cudaStream_t>(stream)>>>(
      iters, static_cast<uint32_t*>(ws));
  return launch_status();
}
