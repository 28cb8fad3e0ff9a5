// C-ABI entry points that compose the kernels: W13, W2 + combine, the whole layer, status.
#include <cuda_runtime.h>

#include <algorithm>

#include "common.cuh"
#include "ptx.cuh"

using namespace moe;

namespace {

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }


}  // namespace

extern "C" const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case MOE_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_TIMEOUT: return "device-side wait timed out";
    case MOE_ERR_DEVICE_INPUT: return "invalid input found on the device (anchor, or a dead row holding slots)";
    default: return "unknown status";
  }
}

extern "C" size_t moe_workspace_bytes(const moe_shape* s) {
  if (!shape_ok(s)) return 0;
  return workspace_layout(s).total;
}

extern "C" int moe_w13_swiglu_grouped(const moe_shape* s, const uint8_t* xq, const uint8_t* xs, const uint8_t* w13,
                                      const uint8_t* w13_s, const int32_t* expert_offsets,
                                      const int32_t* slot_of_row, uint8_t* hq, uint8_t* hs, float* swiglu_debug,
                                      void* ws, size_t ws_bytes, void* stream) {
  if (!s) return MOE_ERR_INVALID_ARG;
  if (!shape_ok(s)) return MOE_ERR_UNSUPPORTED_SHAPE;
  int rc = ws_check(s, ws, ws_bytes);
  if (rc) return rc;
  if (s->T == 0) return MOE_OK;
  if (!xq || !xs || !w13 || !w13_s || !expert_offsets || !slot_of_row || !hq || !hs) return MOE_ERR_INVALID_ARG;
  if (!aligned(xq, 16) || !aligned(xs, 4) || !aligned(w13, 32) || !aligned(w13_s, 16) || !aligned(hq, 16) ||
      !aligned(swiglu_debug, 16))
    return MOE_ERR_INVALID_ARG;
  const Workspace L = workspace_layout(s);
  const bool plan_order = (s->flags & MOE_FLAG_X_PLAN_ORDER) != 0;
  uint8_t* xq_rows = plan_order ? const_cast<uint8_t*>(xq) : ws_ptr<uint8_t>(ws, L.xqp);
  uint8_t* xs_rows = plan_order ? const_cast<uint8_t*>(xs) : ws_ptr<uint8_t>(ws, L.xsp);
  return launch_w13(s, xq, xs, w13, w13_s, expert_offsets, slot_of_row, hq, hs,
                    (s->flags & MOE_FLAG_SWIGLU_DEBUG) ? swiglu_debug : nullptr, ws_ptr<uint32_t>(ws, L.status),
                    xq_rows, xs_rows, plan_order, static_cast<cudaStream_t>(stream));
}

namespace {

// Argument checks of the down projection's GEMM, shared by the entry points that run it.
int w2_args_ok(const uint8_t* hq, const uint8_t* hs, const uint8_t* w2, const uint8_t* w2_s,
               const int32_t* expert_offsets, const int32_t* slot_of_row) {
  if (!hq || !hs || !w2 || !w2_s || !expert_offsets || !slot_of_row) return MOE_ERR_INVALID_ARG;
  if (!aligned(hq, 16) || !aligned(hs, 4) || !aligned(w2, 32) || !aligned(w2_s, 16)) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

// A workspace that only has to hold the status word.
int status_ws_ok(void* ws, size_t ws_bytes) {
  if (!ws || !aligned(ws, 256) || ws_bytes < 256) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

}  // namespace

extern "C" int moe_w2_combine_grouped(const moe_shape* s, const uint8_t* hq, const uint8_t* hs, const uint8_t* w2,
                                      const uint8_t* w2_s, const float* topk_w, const int32_t* expert_offsets,
                                      const int32_t* slot_of_row, const int32_t* row_of_slot, const uint8_t* dead,
                                      uint16_t* out, void* ws, size_t ws_bytes, void* stream) {
  if (!s) return MOE_ERR_INVALID_ARG;
  if (!shape_ok(s)) return MOE_ERR_UNSUPPORTED_SHAPE;
  int rc = ws_check(s, ws, ws_bytes);
  if (rc) return rc;
  if (s->T == 0) return MOE_OK;
  rc = w2_args_ok(hq, hs, w2, w2_s, expert_offsets, slot_of_row);
  if (rc) return rc;
  if (!topk_w || !row_of_slot || !out || !aligned(topk_w, 4) || !aligned(out, 16)) return MOE_ERR_INVALID_ARG;
  const Workspace L = workspace_layout(s);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  float* y = ws_ptr<float>(ws, L.y);
  uint32_t* status = ws_ptr<uint32_t>(ws, L.status);
  rc = launch_w2(s, hq, hs, w2, w2_s, expert_offsets, slot_of_row, y, status, st);
  if (rc) return rc;
  return launch_combine(s, y, topk_w, row_of_slot, out, st, nullptr, dead, status);
}

extern "C" int moe_w2_grouped(const moe_shape* s, const uint8_t* hq, const uint8_t* hs, const uint8_t* w2,
                              const uint8_t* w2_s, const int32_t* expert_offsets, const int32_t* slot_of_row,
                              float* y, void* ws, size_t ws_bytes, void* stream) {
  if (!s) return MOE_ERR_INVALID_ARG;
  if (!shape_ok(s)) return MOE_ERR_UNSUPPORTED_SHAPE;
  int rc = status_ws_ok(ws, ws_bytes);
  if (rc) return rc;
  if (s->T == 0) return MOE_OK;
  rc = w2_args_ok(hq, hs, w2, w2_s, expert_offsets, slot_of_row);
  if (rc) return rc;
  if (!y || !aligned(y, 16)) return MOE_ERR_INVALID_ARG;
  return launch_w2(s, hq, hs, w2, w2_s, expert_offsets, slot_of_row, y, static_cast<uint32_t*>(ws),
                   static_cast<cudaStream_t>(stream));
}

extern "C" int moe_combine(const moe_shape* s, const float* y, const float* topk_w, const int32_t* row_of_slot,
                           const uint8_t* dead, uint16_t* out, void* ws, size_t ws_bytes, void* stream) {
  if (!s) return MOE_ERR_INVALID_ARG;
  if (!shape_ok(s)) return MOE_ERR_UNSUPPORTED_SHAPE;
  int rc = status_ws_ok(ws, ws_bytes);
  if (rc) return rc;
  if (s->T == 0) return MOE_OK;
  if (!y || !topk_w || !row_of_slot || !out || !aligned(y, 16) || !aligned(topk_w, 4) || !aligned(row_of_slot, 4) ||
      !aligned(out, 16))
    return MOE_ERR_INVALID_ARG;
  return launch_combine(s, y, topk_w, row_of_slot, out, static_cast<cudaStream_t>(stream), nullptr, dead,
                        static_cast<uint32_t*>(ws));
}

extern "C" int moe_experts_grouped(const moe_shape* s, const uint8_t* xq, const uint8_t* xs, const uint8_t* w13,
                                   const uint8_t* w13_s, const uint8_t* w2, const uint8_t* w2_s,
                                   const int32_t* expert_offsets, const int32_t* slot_of_row, uint8_t* hq,
                                   uint8_t* hs, float* swiglu_debug, float* y, void* ws, size_t ws_bytes,
                                   void* stream) {
  if (!s) return MOE_ERR_INVALID_ARG;
  if (!shape_ok(s)) return MOE_ERR_UNSUPPORTED_SHAPE;
  int rc = ws_check(s, ws, ws_bytes);
  if (rc) return rc;
  if (s->T == 0) return MOE_OK;
  if (!xq || !xs || !w13 || !w13_s || !hq || !hs || !y) return MOE_ERR_INVALID_ARG;
  rc = w2_args_ok(hq, hs, w2, w2_s, expert_offsets, slot_of_row);
  if (rc) return rc;
  if (!aligned(xq, 16) || !aligned(xs, 4) || !aligned(w13, 32) || !aligned(w13_s, 16) || !aligned(y, 16) ||
      !aligned(swiglu_debug, 16))
    return MOE_ERR_INVALID_ARG;
  const Workspace L = workspace_layout(s);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t* status = ws_ptr<uint32_t>(ws, L.status);
  float* dbg = (s->flags & MOE_FLAG_SWIGLU_DEBUG) ? swiglu_debug : nullptr;
  const bool plan_order = (s->flags & MOE_FLAG_X_PLAN_ORDER) != 0;
  if (fused_gemms_supported(s) && !plan_order) {
    uint32_t* ready = ws_ptr<uint32_t>(ws, L.ready);
    if (cudaMemsetAsync(ready, 0, sizeof(uint32_t) * (s->E + 1), st) != cudaSuccess) return MOE_ERR_CUDA;
    return launch_w13_w2_fused(s, xq, xs, w13, w13_s, w2, w2_s, expert_offsets, slot_of_row, hq, hs, dbg, y, status,
                               ready, st);
  }
  uint8_t* xq_rows = plan_order ? const_cast<uint8_t*>(xq) : ws_ptr<uint8_t>(ws, L.xqp);
  uint8_t* xs_rows = plan_order ? const_cast<uint8_t*>(xs) : ws_ptr<uint8_t>(ws, L.xsp);
  rc = launch_w13(s, xq, xs, w13, w13_s, expert_offsets, slot_of_row, hq, hs, dbg, status, xq_rows, xs_rows,
                  plan_order, st);
  if (rc) return rc;
  return launch_w2(s, hq, hs, w2, w2_s, expert_offsets, slot_of_row, y, status, st);
}

extern "C" int moe_forward(const moe_shape* s, const uint16_t* x, const uint16_t* w_router, const float* bias,
                           const uint8_t* dead, const uint8_t* w13, const uint8_t* w13_s, const uint8_t* w2,
                           const uint8_t* w2_s, uint16_t* out, const moe_intermediates* inter, void* ws,
                           size_t ws_bytes, void* stream) {
  return moe_forward_anchored(s, x, w_router, bias, dead, nullptr, w13, w13_s, w2, w2_s, out, inter, ws, ws_bytes,
                              stream);
}

namespace {

// Shared-expert scratch: identity plan (one expert, row t = token t) and the expert's
// intermediates; its rows enter the combine with weight 1. Every piece 256-byte aligned.
struct SharedWs {
  size_t offsets, slot, hq, hs, y, total;
};

SharedWs shared_layout(int T, int H, int Is) {
  SharedWs w{};
  size_t off = 0;
  auto take = [&](size_t bytes) { size_t o = off; off = align_up(off + (bytes ? bytes : 1), 256); return o; };
  w.offsets = take(2 * 4);
  w.slot = take((size_t)T * 4);
  w.hq = take((size_t)T * Is);
  w.hs = take((size_t)T * hs_pitch(Is));
  w.y = take((size_t)T * H * 4);
  w.total = off;
  return w;
}

__global__ void shared_plan_kernel(int T, int32_t* __restrict__ offsets, int32_t* __restrict__ slot) {
  for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < T; t += gridDim.x * blockDim.x) slot[t] = t;
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    offsets[0] = 0;
    offsets[1] = T;
  }
}

int forward_impl(const moe_shape* s, const uint16_t* x, const uint16_t* w_router, const float* bias,
                 const uint8_t* dead, const int32_t* anchor, const uint8_t* w13, const uint8_t* w13_s,
                 const uint8_t* w2, const uint8_t* w2_s, const moe_shared_expert* shared, uint16_t* out,
                 const moe_intermediates* inter, void* ws, size_t ws_bytes, void* stream, void* side_stream) {
  if (!s) return MOE_ERR_INVALID_ARG;
  if (!aligned(anchor, 4)) return MOE_ERR_INVALID_ARG;
  if (!shape_ok(s)) return MOE_ERR_UNSUPPORTED_SHAPE;
  int rc = ws_check(s, ws, ws_bytes);
  if (rc) return rc;
  moe_shape ss{s->T, s->H, 1, 1, 0, 0};
  if (shared) {
    ss.I = shared->I;
    if (!shape_ok(&ss)) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (!shared->ws || !aligned(shared->ws, 256) || shared->ws_bytes < shared_layout(s->T, s->H, ss.I).total)
      return MOE_ERR_WORKSPACE;
    if (!shared->w13 || !shared->w13_s || !shared->w2 || !shared->w2_s || !aligned(shared->w13, 32) ||
        !aligned(shared->w2, 32) || !aligned(shared->w13_s, 16) || !aligned(shared->w2_s, 16))
      return MOE_ERR_INVALID_ARG;
  }
  if (s->T == 0) return MOE_OK;
  if (!x || !w_router || !bias || !w13 || !w13_s || !w2 || !w2_s || !out) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(w_router, 16) || !aligned(w13, 32) || !aligned(w2, 32) || !aligned(w13_s, 16) ||
      !aligned(w2_s, 16) || !aligned(out, 16))
    return MOE_ERR_INVALID_ARG;
  const Workspace L = workspace_layout(s);
  moe_intermediates im{};
  if (inter) im = *inter;
  if (!aligned(im.xq, 16) || !aligned(im.xs, 4) || !aligned(im.hq, 16) || !aligned(im.hs, 4) ||
      !aligned(im.swiglu, 16) || !aligned(im.topk_idx, 4) || !aligned(im.topk_w, 4))
    return MOE_ERR_INVALID_ARG;
  auto pick = [&](auto* user, size_t off) {
    using Tp = std::remove_pointer_t<decltype(user)>;
    return user ? user : ws_ptr<Tp>(ws, off);
  };
  int32_t* topk_idx = pick(im.topk_idx, L.topk_idx);
  float* topk_w = pick(im.topk_w, L.topk_w);
  int32_t* counts = pick(im.expert_counts, L.counts);
  int32_t* offsets = pick(im.expert_offsets, L.offsets);
  uint8_t* xq = pick(im.xq, L.xq);
  uint8_t* xs = pick(im.xs, L.xs);
  uint8_t* hq = pick(im.hq, L.hq);
  uint8_t* hs = pick(im.hs, L.hs);
  int32_t* slot_of_row = ws_ptr<int32_t>(ws, L.slot_of_row);
  int32_t* row_of_slot = ws_ptr<int32_t>(ws, L.row_of_slot);
  float* y = ws_ptr<float>(ws, L.y);
  uint32_t* status = ws_ptr<uint32_t>(ws, L.status);
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  // decode-sized tiles run W13 and W2 as one persistent launch (its per-expert counters are zeroed
  // by this call's plan kernel); a batch of a few self-routed rows without a shared expert runs
  // the router and then that launch alone, which selects the experts and builds the plan itself
  // (the decode router zeroes the counters)
  uint32_t* ready = ws_ptr<uint32_t>(ws, L.ready);
  const bool fuse_gemms = fused_gemms_supported(s);
  const bool self_plan = fuse_gemms && !shared && !anchor && self_plan_supported(s);
  bool quant_done = false;
  if (self_plan) {
    rc = launch_router_decode_scores(s, x, w_router, bias, ws, st, xq, xs, ready);
    quant_done = true;
  } else {
    rc = launch_route(s, x, w_router, bias, dead, topk_idx, topk_w, counts, offsets, slot_of_row, row_of_slot, ws,
                      st, xq, xs, &quant_done, anchor, fuse_gemms ? ready : nullptr);
  }
  if (rc) return rc;
  uint8_t* xqp = ws_ptr<uint8_t>(ws, L.xqp);
  uint8_t* xsp = ws_ptr<uint8_t>(ws, L.xsp);
  // wide-tile W13 reads the activations in plan order: quantise straight into it (token-order
  // codes are written too when the caller asked for them or the shared expert reads them)
  const bool plan_rows = !quant_done && w13_wants_plan_rows(s);
  if (plan_rows) {
    const bool token_order = im.xq || im.xs || shared;
    rc = launch_quant_mxfp8_plan(s->T, s->H, s->k, x, token_order ? xq : nullptr, token_order ? xs : nullptr,
                                 row_of_slot, xqp, xsp, st);
    if (rc) return rc;
  } else if (!quant_done) {
    rc = launch_quant_mxfp8(s->T, s->H, x, xq, xs, st);
    if (rc) return rc;
  }
  // shared expert ("TP4 serving profile": on a side stream): one dense MXFP8 expert over every
  // row, weight 1, with the same GEMM kernels (identity plan); joined before the combine
  float* y_shared = nullptr;
  cudaEvent_t ev_join = nullptr;
  if (shared) {
    const SharedWs SL = shared_layout(s->T, s->H, ss.I);
    cudaStream_t side = side_stream ? static_cast<cudaStream_t>(side_stream) : st;
    if (side != st) {
      cudaEvent_t ev_fork = nullptr;
      if (cudaEventCreateWithFlags(&ev_fork, cudaEventDisableTiming) != cudaSuccess) return MOE_ERR_CUDA;
      const bool ok = cudaEventRecord(ev_fork, st) == cudaSuccess && cudaStreamWaitEvent(side, ev_fork, 0) == cudaSuccess;
      cudaEventDestroy(ev_fork);
      if (!ok) return MOE_ERR_CUDA;
    }
    int32_t* s_off = ws_ptr<int32_t>(shared->ws, SL.offsets);
    int32_t* s_slot = ws_ptr<int32_t>(shared->ws, SL.slot);
    uint8_t* s_hq = ws_ptr<uint8_t>(shared->ws, SL.hq);
    uint8_t* s_hs = ws_ptr<uint8_t>(shared->ws, SL.hs);
    y_shared = ws_ptr<float>(shared->ws, SL.y);
    const int blocks = (int)std::min<long long>((s->T + 255) / 256, (long long)num_sms() * 4);
    shared_plan_kernel<<<blocks, 256, 0, side>>>(s->T, s_off, s_slot);
    rc = launch_status();
    if (rc) return rc;
    rc = launch_w13(&ss, xq, xs, shared->w13, shared->w13_s, s_off, s_slot, s_hq, s_hs, nullptr, status, xq, xs,
                    true, side, true);
    if (rc) return rc;
    rc = launch_w2(&ss, s_hq, s_hs, shared->w2, shared->w2_s, s_off, s_slot, y_shared, status, side, true);
    if (rc) return rc;
    if (side != st) {
      if (cudaEventCreateWithFlags(&ev_join, cudaEventDisableTiming) != cudaSuccess) return MOE_ERR_CUDA;
      if (cudaEventRecord(ev_join, side) != cudaSuccess) {
        cudaEventDestroy(ev_join);
        return MOE_ERR_CUDA;
      }
    }
  }
  // with no shared expert to add, the one-launch GEMMs also run the combine at their end
  const bool fused_combine = fuse_gemms && !shared;
  if (fuse_gemms) {
    const SelfPlanArgs sp{ws_ptr<float2>(ws, L.selrep), dead, topk_idx, topk_w, counts, offsets, slot_of_row,
                          row_of_slot};
    rc = launch_w13_w2_fused(s, xq, xs, w13, w13_s, w2, w2_s, offsets, slot_of_row, hq, hs, im.swiglu, y, status,
                             ready, st, fused_combine ? topk_w : nullptr, fused_combine ? row_of_slot : nullptr,
                             fused_combine ? out : nullptr, self_plan ? &sp : nullptr);
  } else {
    rc = launch_w13(s, xq, xs, w13, w13_s, offsets, slot_of_row, hq, hs, im.swiglu, status, xqp, xsp, plan_rows, st);
    if (!rc) rc = launch_w2(s, hq, hs, w2, w2_s, offsets, slot_of_row, y, status, st);
  }
  if (ev_join) {
    if (!rc && cudaStreamWaitEvent(st, ev_join, 0) != cudaSuccess) rc = MOE_ERR_CUDA;
    cudaEventDestroy(ev_join);
  }
  if (rc) return rc;
  if (fused_combine) return MOE_OK;
  return launch_combine(s, y, topk_w, row_of_slot, out, st, y_shared, dead, status);
}

}  // namespace

extern "C" int moe_forward_anchored(const moe_shape* s, const uint16_t* x, const uint16_t* w_router,
                                    const float* bias, const uint8_t* dead, const int32_t* anchor,
                                    const uint8_t* w13, const uint8_t* w13_s, const uint8_t* w2, const uint8_t* w2_s,
                                    uint16_t* out, const moe_intermediates* inter, void* ws, size_t ws_bytes,
                                    void* stream) {
  return forward_impl(s, x, w_router, bias, dead, anchor, w13, w13_s, w2, w2_s, nullptr, out, inter, ws, ws_bytes,
                      stream, nullptr);
}

extern "C" size_t moe_shared_workspace_bytes(const moe_shape* s, int32_t I_shared) {
  if (!s || !shape_ok(s)) return 0;
  moe_shape ss{s->T, s->H, 1, 1, I_shared, 0};
  if (!shape_ok(&ss)) return 0;
  return shared_layout(s->T, s->H, I_shared).total;
}

extern "C" int moe_forward_shared(const moe_shape* s, const uint16_t* x, const uint16_t* w_router, const float* bias,
                                  const uint8_t* dead, const int32_t* anchor, const uint8_t* w13,
                                  const uint8_t* w13_s, const uint8_t* w2, const uint8_t* w2_s,
                                  const moe_shared_expert* shared, uint16_t* out, const moe_intermediates* inter,
                                  void* ws, size_t ws_bytes, void* stream, void* side_stream) {
  if (!shared) return MOE_ERR_INVALID_ARG;
  return forward_impl(s, x, w_router, bias, dead, anchor, w13, w13_s, w2, w2_s, shared, out, inter, ws, ws_bytes,
                      stream, side_stream);
}

extern "C" int moe_check_device_status(void* ws, void* stream) {
  if (!ws) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t h = 0;
  if (cudaMemcpyAsync(&h, ws, 4, cudaMemcpyDeviceToHost, st) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
  if (h != 0) {
    if (cudaMemsetAsync(ws, 0, 4, st) != cudaSuccess || cudaStreamSynchronize(st) != cudaSuccess)
      return MOE_ERR_CUDA;
    return h == DEV_BAD_INPUT ? MOE_ERR_DEVICE_INPUT : MOE_ERR_TIMEOUT;
  }
  return MOE_OK;
}

// ---------------------------------------------------------------------------------------------
// Self-test of the bounded-wait machinery: one thread waits on an mbarrier that nothing ever
// arrives at, with a caller-chosen limit. The wait expires, records its code in the status word,
// and the kernel returns normally -- the context stays usable.
// ---------------------------------------------------------------------------------------------
#include "ptx.cuh"

namespace moe {
__global__ void selftest_timeout_kernel(uint32_t* status, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar, 1);
    mbar_fence_init();
    mbar_wait(&bar, 0, limit_ns, &abort_flag, status, DEV_TIMEOUT_FULL);
  }
}
}  // namespace moe

extern "C" int moe_selftest_timeout(void* ws, uint64_t limit_ns, void* stream) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255)) return MOE_ERR_WORKSPACE;
  if (limit_ns > 2000000000ull) return MOE_ERR_INVALID_ARG;
  selftest_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(static_cast<uint32_t*>(ws), limit_ns);
  return launch_status();
}
