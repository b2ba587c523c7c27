// Commit-aware KV tiering ("Resource-Efficient Speculative Decoding for
// Long-Context LLM Serving", section 4.1, Eqs. 4-5): the three regions of one
// request's Target KV, the migration endpoint, the asynchronous migration of
// [H, E) to host memory, and rollback that never reaches the CPU history.
//
// The state transitions are host-only integer logic; svx_tier_migrate adds the
// device-to-host copy of the interval and svx_tier_poll advances H once that
// copy has completed.
#include <cuda_runtime.h>

#include <algorithm>

#include "svx.h"

namespace {

bool valid(const svx_tier_state* s) { return s && 0 <= s->H && s->H <= s->C && s->C <= s->L; }

int64_t endpoint(int64_t H, int64_t C, int64_t T, int64_t g) {
  return std::max<int64_t>(H, g * (std::max<int64_t>(0, C - T) / g));
}

}  // namespace

extern "C" {

svx_status svx_migration_endpoint(int64_t H, int64_t C, int64_t T, int64_t g, int64_t* E_out) {
  if (!E_out || g < 1 || T < 0 || H < 0 || C < H || H % g) return SVX_ERR_INVALID_ARG;
  *E_out = endpoint(H, C, T, g);
  return SVX_OK;
}

svx_status svx_tier_round(svx_tier_state* s, int64_t C, int64_t L) {
  if (!valid(s) || C < s->C || L < C) return SVX_ERR_INVALID_ARG;
  s->C = C;
  s->L = L;
  return SVX_OK;
}

svx_status svx_tier_plan(svx_tier_state* s, int64_t T, int64_t g, int64_t* begin, int64_t* end) {
  if (!valid(s) || !begin || !end || g < 1 || T < 0 || s->H % g) return SVX_ERR_INVALID_ARG;
  *begin = *end = s->H;
  if (s->pending >= 0) return SVX_OK;  // one migration at a time
  const int64_t E = endpoint(s->H, s->C, T, g);
  if (E > s->H) {
    *end = E;
    s->pending = E;
  }
  return SVX_OK;
}

svx_status svx_tier_complete(svx_tier_state* s) {
  if (!valid(s)) return SVX_ERR_INVALID_ARG;
  if (s->event) return SVX_ERR_BAD_STATE;  // the library's own copy is in flight: poll or release it
  if (s->pending >= 0) {
    s->H = s->pending;
    s->pending = -1;
  }
  return SVX_OK;
}

svx_status svx_tier_commit(svx_tier_state* s, int64_t C_new, int64_t* rel_begin, int64_t* rel_end) {
  if (!valid(s) || !rel_begin || !rel_end || C_new < s->C || C_new > s->L) return SVX_ERR_INVALID_ARG;
  if (C_new < s->H) return SVX_ERR_BAD_STATE;  // unreachable while H <= C_r <= C'_r
  *rel_begin = C_new;
  *rel_end = s->L;
  s->C = s->L = C_new;
  return SVX_OK;
}

svx_status svx_tier_migrate(svx_tier_state* s, int64_t T, int64_t g, int64_t row_bytes, const void* k_dev_at_H,
                            const void* v_dev_at_H, void* k_host, void* v_host, void* stream, int64_t* E_out) {
  if (!valid(s) || !E_out || row_bytes <= 0) return SVX_ERR_INVALID_ARG;
  if (s->event) return SVX_ERR_BAD_STATE;  // the previous migration has not been polled to completion
  int64_t b = 0, e = 0;
  svx_status st = svx_tier_plan(s, T, g, &b, &e);
  if (st != SVX_OK) return st;
  *E_out = e;
  if (e == b) return SVX_OK;
  if (!k_dev_at_H || !v_dev_at_H || !k_host || !v_host) {
    s->pending = -1;
    return SVX_ERR_INVALID_ARG;
  }
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const size_t bytes = static_cast<size_t>(e - b) * static_cast<size_t>(row_bytes);
  cudaEvent_t ev = nullptr;
  if (cudaEventCreateWithFlags(&ev, cudaEventDisableTiming) != cudaSuccess ||
      cudaMemcpyAsync(static_cast<char*>(k_host) + b * row_bytes, k_dev_at_H, bytes, cudaMemcpyDeviceToHost, cs) !=
          cudaSuccess ||
      cudaMemcpyAsync(static_cast<char*>(v_host) + b * row_bytes, v_dev_at_H, bytes, cudaMemcpyDeviceToHost, cs) !=
          cudaSuccess ||
      cudaEventRecord(ev, cs) != cudaSuccess) {
    cudaGetLastError();
    if (ev) cudaEventDestroy(ev);
    s->pending = -1;
    return SVX_ERR_CUDA;
  }
  s->event = ev;
  return SVX_OK;
}

svx_status svx_tier_poll(svx_tier_state* s, int32_t* done) {
  if (!valid(s) || !done) return SVX_ERR_INVALID_ARG;
  *done = 1;
  if (!s->event) return SVX_OK;
  cudaEvent_t ev = static_cast<cudaEvent_t>(s->event);
  const cudaError_t e = cudaEventQuery(ev);
  if (e == cudaErrorNotReady) {
    *done = 0;
    return SVX_OK;
  }
  cudaEventDestroy(ev);
  s->event = nullptr;
  if (e != cudaSuccess) {
    cudaGetLastError();
    s->pending = -1;  // the copy failed: H stays where it was
    return SVX_ERR_CUDA;
  }
  return svx_tier_complete(s);  // H advances only now that the data is in host memory
}

svx_status svx_tier_release(svx_tier_state* s) {
  if (!s) return SVX_ERR_INVALID_ARG;
  if (s->event) {
    cudaEvent_t ev = static_cast<cudaEvent_t>(s->event);
    const cudaError_t e = cudaEventSynchronize(ev);
    cudaEventDestroy(ev);
    s->event = nullptr;
    if (e != cudaSuccess) {
      cudaGetLastError();
      s->pending = -1;
      return SVX_ERR_CUDA;
    }
    return svx_tier_complete(s);
  }
  return SVX_OK;
}

}  // extern "C"
