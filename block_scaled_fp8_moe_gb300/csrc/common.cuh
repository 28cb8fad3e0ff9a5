// Host-side helpers shared by the translation units of libmoe: shape checks, workspace layout,
// launch-error mapping.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include <map>
#include <mutex>
#include <utility>

#include "../../include/moe.h"

namespace moe {

constexpr int kRouterChunk = 64;       // fixed reduction chunk of the router logits
constexpr int kPlanBlock = 256;        // tokens per plan-count block
constexpr int kMaxE = 1024;
constexpr int kMaxK = 32;
// One-launch decode layer that routes itself: up to 12 rows (a warp of the fused GEMM CTA selects
// one or two of them; all 8 warps taking two, at 16 rows, measured slower than the plan kernel),
// every expert's key in 8 registers per lane of the selecting warp
constexpr int kSelfPlanMaxT = 12;
constexpr int kSelfPlanMaxE = 256;
constexpr int kSelfPlanNI = kSelfPlanMaxE / 32;
// ... reading its rows' (key, score) pairs from one of this many copies (CTA b: copy b mod n), so
// that the GPU's CTAs do not all queue on the same few L2 lines
constexpr int kSelfPlanReplicas = 8;
constexpr int kTileK = 128;            // K elements per packed tile / pipeline stage
constexpr int kTileRows = 128;         // weight rows per packed tile
constexpr int kTileCodeBytes = kTileRows * kTileK / 2;   // 8192
constexpr int kTileScaleBytes = 512;

__host__ __device__ inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

inline bool shape_ok(const moe_shape* s) {
  if (!s) return false;
  if (s->T < 0 || s->H <= 0 || s->E <= 0 || s->k <= 0 || s->I <= 0) return false;
  if (s->H % 128 || s->I % 64) return false;
  if (s->k > kMaxK || s->k > s->E || s->E > kMaxE) return false;
  if (s->H > 16384 || s->I > 16384) return false;
  if ((int64_t)s->T * s->k > (int64_t)1 << 30) return false;
  return true;
}

inline int hs_pitch(int I) { return (int)(align_up((size_t)I, 128) / 32); }

// Workspace carve-up. Every piece 256-byte aligned; the status word sits at offset 0.
struct Workspace {
  size_t status, score, key, cnt, base, rank;                  // router scratch
  size_t topk_idx, topk_w, counts, offsets, slot_of_row, row_of_slot;
  size_t xq, xs, hq, hs, y;                                    // forward intermediates
  size_t xqp, xsp;                                             // plan-order copy of xq / xs
  size_t xnorm, wnorm, cand, ncand;                            // router screen
  size_t ready;                                                // per-expert W13 tile counters
  size_t selrep;                                               // self-routed batches: (key, score) copies
  size_t total;
};

inline Workspace workspace_layout(const moe_shape* s) {
  Workspace w{};
  size_t T = (size_t)s->T, E = (size_t)s->E, k = (size_t)s->k, H = (size_t)s->H, I = (size_t)s->I;
  size_t nb = (T + kPlanBlock - 1) / kPlanBlock;
  size_t off = 0;
  auto take = [&](size_t bytes) { size_t o = off; off = align_up(off + (bytes ? bytes : 1), 256); return o; };
  w.status = take(256);
  w.score = take(T * E * 4);
  w.key = take(T * E * 4);
  w.cnt = take(nb * E * 4);
  w.base = take(nb * E * 4);
  w.rank = take(T * k * 4);
  w.topk_idx = take(T * k * 4);
  w.topk_w = take(T * k * 4);
  w.counts = take(E * 4);
  w.offsets = take((E + 1) * 4);
  w.slot_of_row = take(T * k * 4);
  w.row_of_slot = take(T * k * 4);
  w.xq = take(T * H);
  w.xs = take(T * H / 32);
  w.hq = take(T * k * I);
  w.hs = take(T * k * (size_t)hs_pitch((int)I));
  w.y = take(T * k * H * 4);
  w.xqp = take(T * k * H);
  w.xsp = take(T * k * H / 32);
  w.xnorm = take(T * 4);
  w.wnorm = take(E * 4);
  w.cand = take(T * 64 * 4);
  w.ncand = take(T * 4);
  w.ready = take((E + 1) * 4);
  w.selrep = take((T <= (size_t)kSelfPlanMaxT && E <= (size_t)kSelfPlanMaxE) ? kSelfPlanReplicas * T * E * 8 : 0);
  w.total = off;
  return w;
}

inline int ws_check(const moe_shape* s, void* ws, size_t ws_bytes) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255)) return MOE_ERR_WORKSPACE;
  if (ws_bytes < workspace_layout(s).total) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

template <typename T>
inline T* ws_ptr(void* ws, size_t off) { return reinterpret_cast<T*>(static_cast<char*>(ws) + off); }

inline int launch_status() {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

constexpr int kMaxDevices = 64;

inline int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  return dev;
}

// Per-device properties, read once per device (every GPU of a process gets its own entry).
struct DeviceProps {
  int sms = 0, smem_per_sm = 0, smem_reserved = 0;
};

inline const DeviceProps& device_props() {
  static std::mutex mu;
  static DeviceProps props[kMaxDevices];
  const int dev = current_device();
  std::lock_guard<std::mutex> lock(mu);
  DeviceProps& p = props[dev];
  if (!p.sms) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
    if (cudaDeviceGetAttribute(&p.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
        p.smem_per_sm <= 0)
      p.smem_per_sm = 228 * 1024;
    if (cudaDeviceGetAttribute(&p.smem_reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess)
      p.smem_reserved = 1024;
    p.sms = n;
  }
  return p;
}

inline int num_sms() { return device_props().sms; }

// CTAs of `smem_bytes` dynamic shared memory that fit on one SM, capped at `cap` (the per-SM
// shared-memory capacity minus the per-block reservation, as the device reports them).
inline int ctas_per_sm_by_smem(size_t smem_bytes, int cap) {
  const DeviceProps& p = device_props();
  int n = (int)((size_t)p.smem_per_sm / (smem_bytes + (size_t)p.smem_reserved));
  if (n > cap) n = cap;
  return n < 1 ? 1 : n;
}

// Raises a kernel's dynamic shared-memory limit to at least `bytes` on the current device. The
// attribute belongs to the (kernel, device) pair, so each GPU a process uses is set up on its first
// launch there; later calls only look the pair up.
inline int ensure_smem_limit(const void* kern, int bytes) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, int> done;
  const std::pair<const void*, int> key(kern, current_device());
  std::lock_guard<std::mutex> lock(mu);
  auto it = done.find(key);
  if (it != done.end() && it->second >= bytes) return MOE_OK;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  done[key] = bytes;
  return MOE_OK;
}

// Launch with the programmatic-stream-serialization attribute: the kernel may begin while the
// previous kernel on `st` finishes (it calls pdl_wait() before reading anything produced upstream).
template <typename... KArgs, typename... Args>
inline int launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

// Internal launchers (defined in the .cu files), all asynchronous on `st`.
int launch_quant_mxfp8(int rows, int cols, const uint16_t* x, uint8_t* q, uint8_t* s, cudaStream_t st);
// Quantises x and writes codes/scales to plan rows row_of_slot[t k + j] of qp/sp (q/s nullable).
int launch_quant_mxfp8_plan(int rows, int cols, int k, const uint16_t* x, uint8_t* q, uint8_t* s,
                            const int32_t* row_of_slot, uint8_t* qp, uint8_t* sp, cudaStream_t st);
// True when W13 runs wide token tiles, whose activation operand is read in plan order.
bool w13_wants_plan_rows(const moe_shape* s);
// When xq/xs are given and the small-batch router runs, it also writes the MXFP8 quantisation of x
// and sets *quant_done. anchor (nullable): rows that reuse another row's experts. ready (nullable):
// E + 1 counters the plan kernel zeroes for the one-launch W13 + W2 GEMM.
int launch_route(const moe_shape* s, const uint16_t* x, const uint16_t* wr, const float* bias, const uint8_t* dead,
                 int32_t* topk_idx, float* topk_w, int32_t* counts, int32_t* offsets, int32_t* slot_of_row,
                 int32_t* row_of_slot, void* ws, cudaStream_t st, uint8_t* xq, uint8_t* xs, bool* quant_done,
                 const int32_t* anchor, uint32_t* ready);
// The decode router alone (scores, keys, kSelfPlanReplicas copies of the (key, score) pairs in the
// workspace, and the MXFP8 quantisation of x into xq/xs), for a layer call whose fused GEMM routes
// itself (self_plan_supported); it also zeroes the E + 1 counters in ready.
bool self_plan_supported(const moe_shape* s);
int launch_router_decode_scores(const moe_shape* s, const uint16_t* x, const uint16_t* wr, const float* bias, void* ws,
                                cudaStream_t st, uint8_t* xq, uint8_t* xs, uint32_t* ready);
// The routing plan a self-routing fused GEMM builds (every CTA in shared memory) from the router's
// (key, score) pairs [kSelfPlanReplicas][T][E], and the arrays its CTA 0 writes it to.
struct SelfPlanArgs {
  const float2* sel;
  const uint8_t* dead;
  int32_t* topk_idx;
  float* topk_w;
  int32_t* counts;
  int32_t* offsets;
  int32_t* slot_of_row;
  int32_t* row_of_slot;
};
// W13 then W2 in one persistent launch, for decode-sized token tiles (fused_gemms_supported):
// writes hq/hs (and dbg) like launch_w13 and y like launch_w2, and with out non-null also the
// combine's output, like launch_combine without a shared expert or dead mask. ready: E + 1
// counters, zeroed by the kernel before it in this layer call. With sp non-null (requires out and
// self_plan_supported) the launch routes itself and offsets / slot_of_row / topk_w / row_of_slot
// are not read.
bool fused_gemms_supported(const moe_shape* s);
int launch_w13_w2_fused(const moe_shape* s, const uint8_t* xq, const uint8_t* xs, const uint8_t* w13,
                        const uint8_t* w13s, const uint8_t* w2, const uint8_t* w2s, const int32_t* offsets,
                        const int32_t* slot_of_row, uint8_t* hq, uint8_t* hs, float* dbg, float* y, uint32_t* status,
                        uint32_t* ready, cudaStream_t st, const float* topk_w = nullptr,
                        const int32_t* row_of_slot = nullptr, uint16_t* out = nullptr,
                        const SelfPlanArgs* sp = nullptr);
int launch_w13(const moe_shape* s, const uint8_t* xq, const uint8_t* xs, const uint8_t* w13, const uint8_t* w13s,
               const int32_t* offsets, const int32_t* slot_of_row, uint8_t* hq, uint8_t* hs, float* dbg,
               uint32_t* status, uint8_t* xq_plan, uint8_t* xs_plan, bool plan_rows_ready, cudaStream_t st,
               bool fp8_weights = false);
// y: plan-order rows W2[e] h^ (fp32, before the routing weight)
int launch_w2(const moe_shape* s, const uint8_t* hq, const uint8_t* hs, const uint8_t* w2, const uint8_t* w2s,
              const int32_t* offsets, const int32_t* slot_of_row, float* y, uint32_t* status, cudaStream_t st,
              bool fp8_weights = false);
// out[t] = bf16(((w_0 y[r_0] + w_1 y[r_1]) + ...)), r_j = row_of_slot[t k + j], w_j = topk_w[t k + j];
// y_shared (nullable): a per-token row added after the routed slots (the shared expert); dead
// (nullable): rows forced to +0.0, a forced row that holds slots is recorded in *status
int launch_combine(const moe_shape* s, const float* y, const float* topk_w, const int32_t* row_of_slot,
                   uint16_t* out, cudaStream_t st, const float* y_shared, const uint8_t* dead, uint32_t* status);
// Large-T router: certified tensor-core screen + exact recompute of the surviving experts; writes
// the same score/key rows as the exact router for every expert that can be selected.
bool router_screen_supported(const moe_shape* s);
int launch_router_screen(const moe_shape* s, const uint16_t* x, const uint16_t* wr, const float* bias, void* ws,
                         float* score, float* key, cudaStream_t st, const int32_t* anchor);

}  // namespace moe
