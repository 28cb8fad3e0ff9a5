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
constexpr int kProbeSmem = 200 * 1024;
constexpr uint64_t kProbeWaitNs = 1000000000ull;

__device__ __forceinline__ uint32_t probe_hash(uint32_t v) {
  v ^= v >> 16;
  v *= 0x7feb352du;
  v ^= v >> 15;
  v *= 0x846ca68bu;
  v ^= v >> 16;
  return v;
}

// mode bit 0: the MMAs of consecutive K-chunks read 4 different operand buffers in turn (as a
//             pipeline's stages do) instead of one;
//      bit 1: each K-chunk of 4 MMAs is preceded by the scale copies the grouped GEMMs issue (one
//             A atom, one B atom per 128 columns) into a ring of TMEM slots;
//      bit 2: N = 224 (the widest gate/up tile) instead of 256.
constexpr int kProbeBufs = 4;

__global__ void __launch_bounds__(kProbeThreads, 1) mma_rate_probe_kernel(int iters, int mode, uint32_t* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr int kBuf = 128 * 128 + kProbeN * 128;      // A tile + B tile (48 KB)
  uint8_t* sSF = base + kProbeBufs * kBuf;             // A scale atom (512 B), then two B scale atoms
  uint64_t* done = reinterpret_cast<uint64_t*>(sSF + 3 * 512);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  const int warp = threadIdx.x >> 5;
  const int nbuf = (mode & 1) ? kProbeBufs : 1;
  const bool copies = (mode & 2) != 0;
  const uint32_t N = (mode & 4) ? 224 : kProbeN;

  // operands: pseudo-random bytes (every E2M1 code is finite; E4M3 NaN codes are moved to the
  // neighbouring finite code), scales 2^0
  for (int i = threadIdx.x; i < nbuf * kBuf; i += kProbeThreads) {
    uint8_t b = (uint8_t)probe_hash((uint32_t)i * 2654435761u + blockIdx.x);
    if ((i % kBuf) >= 128 * 128 && (b & 0x7f) == 0x7f) b -= 1;
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
    // TMEM: accumulator at column 0 (N columns), scale slots of 12 columns from column 256
    const uint32_t sf0 = tmem + 256;
    tc_cp_32x128b_warpx4(sf0, smem_desc(smem_u32(sSF), 16, 128, 0));
    tc_cp_32x128b_warpx4(sf0 + 4, smem_desc(smem_u32(sSF + 512), 16, 128, 0));
    tc_cp_32x128b_warpx4(sf0 + 8, smem_desc(smem_u32(sSF + 1024), 16, 128, 0));
    const uint32_t idesc0 = idesc_mxf8f6f4(5 /*E2M1*/, 0 /*E4M3*/, 128, N, 0, 0);
    for (int it = 0; it < iters; ++it) {
      const int kb = it & 3;
      const int chunk = it >> 2;
      const uint32_t slot = copies ? (uint32_t)(chunk % 16) * 12 : 0;
      if (copies && kb == 0) {
        tc_cp_32x128b_warpx4(sf0 + slot, smem_desc(smem_u32(sSF), 16, 128, 0));
        tc_cp_32x128b_warpx4(sf0 + slot + 4, smem_desc(smem_u32(sSF + 512), 16, 128, 0));
        tc_cp_32x128b_warpx4(sf0 + slot + 8, smem_desc(smem_u32(sSF + 1024), 16, 128, 0));
      }
      const uint8_t* buf = base + (chunk % nbuf) * kBuf;
      const uint32_t a0 = smem_u32(buf), b0 = smem_u32(buf + 128 * 128);
      const uint32_t id = idesc0 | ((uint32_t)kb << 4) | ((uint32_t)kb << 29);
      mma_mxf8f6f4(tmem, smem_desc(a0 + kb * 32, 16, 1024, 2), smem_desc(b0 + kb * 32, 16, 1024, 2), id, sf0 + slot,
                   sf0 + slot + 4, it > 0 ? 1u : 0u);
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

extern "C" int moe_probe_mma_rate(int32_t iters, int32_t mode, int32_t* ctas, int64_t* flops, void* ws,
                                  size_t ws_bytes, void* stream) {
  if (iters <= 0 || iters > (1 << 24) || mode < 0 || mode > 7 || !ctas || !flops) return MOE_ERR_INVALID_ARG;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255) || ws_bytes < 256) return MOE_ERR_WORKSPACE;
  if (ensure_smem_limit((const void*)mma_rate_probe_kernel, kProbeSmem)) return MOE_ERR_CUDA;
  const int grid = num_sms();
  *ctas = grid;
  *flops = 2LL * 128 * ((mode & 4) ? 224 : kProbeN) * 32 * (int64_t)iters * grid;
  mma_rate_probe_kernel<<<grid, kProbeThreads, kProbeSmem, static_cast<cudaStream_t>(stream)>>>(
      iters, mode, static_cast<uint32_t*>(ws));
  return launch_status();
}
