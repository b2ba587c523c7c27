// svx_verify_static: one whole verification round over device-resident KV that
// allocates no device memory.  Its fp32 state workspace and the device error
// word live in a file-scope
// `static __device__` array of fixed size, which every GPU that loads this
// library holds until the process exits.
//
// Who needs it: callers that cannot call cudaMalloc once they are running - an
// inference engine whose memory manager owns all device memory after start-up
// and forbids any other allocation, or a latency-critical decode loop where an
// allocation (and the device synchronisation cudaFree implies) is not
// acceptable.  Such callers pass inputs and outputs; this entry point only
// launches the library's existing kernels on their stream.
//
// Host code must not pass `g_static_scratch` itself to a kernel: on the host
// that name is only a stand-in, not a device address.  The device address is
// fetched once per device with cudaGetSymbolAddress (with that device current)
// and cached.
#include <cstdarg>
#include <cstdio>
#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>

#include "svx.h"
#include "svx_internal.h"

namespace svx {
void set_thread_error(const char* msg);  // svx_runtime.cu: message for svx_last_error(NULL)
}

namespace {

constexpr size_t kScratchBytes = SVX_STATIC_SCRATCH_BYTES;
constexpr size_t kErrOffset = 0;
constexpr size_t kStateOffset = 256;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_static_scratch[kScratchBytes];

struct StaticDevice {
  std::mutex mu;
  bool ready = false;
  unsigned char* ptr = nullptr;  // device address of g_static_scratch on this device
  uint32_t epoch = 0;
};
StaticDevice g_devices[kMaxDevices];

svx_status fail(svx_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  svx::set_thread_error(buf);
  return st;
}

bool is_device_ptr(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" svx_status svx_verify_static(int32_t n_req, int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim,
                                        int32_t n_query, const void* q_dev, const int64_t* hist_len_host,
                                        const void* const* k_hist_dev, const void* const* v_hist_dev,
                                        const void* k_cand_dev, const void* v_cand_dev, const int32_t* parent_host,
                                        float scale, void* o_dev, float* lse_dev, void* stream) {
  // ---- arguments (no CUDA call before the size check)
  if (n_req < 1 || n_req > svx::kMaxReq) return fail(SVX_ERR_INVALID_ARG, "n_req must be in [1, %d]", svx::kMaxReq);
  if (n_kv_heads < 1 || n_q_heads < n_kv_heads || n_q_heads % n_kv_heads)
    return fail(SVX_ERR_INVALID_ARG, "n_q_heads must be a positive multiple of n_kv_heads");
  if (head_dim != 64 && head_dim != 128) return fail(SVX_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
  if (n_query < 1 || n_query > 32) return fail(SVX_ERR_INVALID_ARG, "n_query must be in [1, 32]");
  if (!hist_len_host || !q_dev || !o_dev || !lse_dev || !aligned16(q_dev) || !aligned16(o_dev) ||
      !aligned16(lse_dev))
    return fail(SVX_ERR_INVALID_ARG, "q, o, lse must be 16-byte aligned device pointers and hist_len non-NULL");
  if ((k_cand_dev == nullptr) != (v_cand_dev == nullptr))
    return fail(SVX_ERR_INVALID_ARG, "give both candidate k and v, or neither");
  const int64_t rows = static_cast<int64_t>(n_req) * n_q_heads * n_query;
  const size_t need = kStateOffset + static_cast<size_t>(svx::kHistSlots) * static_cast<size_t>(rows) *
                                         (sizeof(svx::RowState) + sizeof(float) * head_dim);
  if (need > kScratchBytes)
    return fail(SVX_ERR_INVALID_ARG,
                "round needs %zu bytes of static scratch (%lld query rows); the limit is %zu bytes "
                "(SVX_STATIC_SCRATCH_BYTES): use the context API for rounds this large",
                need, static_cast<long long>(rows), kScratchBytes);
  for (int b = 0; b < n_req; ++b) {
    if (hist_len_host[b] < 0 || hist_len_host[b] > 0x7fffffff)
      return fail(SVX_ERR_INVALID_ARG, "hist_len[%d] must be in [0, 2^31)", b);
    if (hist_len_host[b] > 0 && (!k_hist_dev || !v_hist_dev || !k_hist_dev[b] || !v_hist_dev[b] ||
                                 !aligned16(k_hist_dev[b]) || !aligned16(v_hist_dev[b])))
      return fail(SVX_ERR_INVALID_ARG, "history of request %d needs 16-byte aligned k and v pointers", b);
  }
  if (k_cand_dev && (!aligned16(k_cand_dev) || !aligned16(v_cand_dev)))
    return fail(SVX_ERR_INVALID_ARG, "candidate k/v must be 16-byte aligned");
  static thread_local uint32_t vis_check[svx::kMaxReq * 32];  // validation only
  if (k_cand_dev && svx_candidate_masks(n_req, n_query, parent_host, vis_check) != SVX_OK)
    return fail(SVX_ERR_INVALID_ARG, "invalid token-tree parents");

  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return fail(SVX_ERR_CUDA, "no usable current CUDA device");
  }
  if (!is_device_ptr(q_dev) || !is_device_ptr(o_dev) || !is_device_ptr(lse_dev) ||
      (k_cand_dev && (!is_device_ptr(k_cand_dev) || !is_device_ptr(v_cand_dev))))
    return fail(SVX_ERR_INVALID_ARG, "q, o, lse and candidate k/v must be device memory");
  for (int b = 0; b < n_req; ++b)
    if (hist_len_host[b] > 0 && (!is_device_ptr(k_hist_dev[b]) || !is_device_ptr(v_hist_dev[b])))
      return fail(SVX_ERR_INVALID_ARG, "history of request %d must be device memory", b);

  StaticDevice& sd = g_devices[dev];
  std::lock_guard<std::mutex> lock(sd.mu);
  // ---- set-up, once per device, with that device current: the array's device address, zeroed
  if (!sd.ready) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) return fail(SVX_ERR_CUDA, "cudaGetSymbolAddress failed: %s", cudaGetErrorString(e));
    e = cudaMemset(p, 0, kScratchBytes);  // epoch 0 = never written; error word 0
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return fail(SVX_ERR_CUDA, "static scratch set-up failed: %s", cudaGetErrorString(e));
    sd.ptr = static_cast<unsigned char*>(p);
    sd.ready = true;
  }
  sd.epoch = sd.epoch == 0xffffffffu ? 1u : sd.epoch + 1u;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int num_sms = 0;
  if (cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return fail(SVX_ERR_CUDA, "cannot read the SM count");

  int* d_err = reinterpret_cast<int*>(sd.ptr + kErrOffset);
  svx::RowState* ws_h = reinterpret_cast<svx::RowState*>(sd.ptr + kStateOffset);
  float* ws_a = reinterpret_cast<float*>(sd.ptr + kStateOffset +
                                         static_cast<size_t>(svx::kHistSlots) * rows * sizeof(svx::RowState));
  const int G = n_q_heads / n_kv_heads;
  const int R = G * n_query;
  const float sc = scale > 0.f ? scale : 1.0f / sqrtf(static_cast<float>(head_dim));
  uint32_t slot_mask[svx::kMaxReq] = {};

  svx::ChunkParams p;
  std::memset(&p, 0, sizeof(p));
  p.q = static_cast<const __nv_bfloat16*>(q_dev);
  p.ws_h = ws_h;
  p.ws_a = ws_a;
  p.err = d_err;
  p.slot_stride = rows;
  p.q_rows = rows;
  p.q_scale = sc * 1.4426950408889634f;
  p.epoch = sd.epoch;
  p.n_q_heads = n_q_heads;
  p.n_kv_heads = n_kv_heads;
  p.group = G;
  p.n_query = n_query;

  // ---- history: one in-place part per request, batches of kMaxPartsPerLaunch
  int reqs[svx::kMaxReq];
  int n_hist = 0;
  for (int b = 0; b < n_req; ++b)
    if (hist_len_host[b] > 0) reqs[n_hist++] = b;
  for (int i0 = 0; i0 < n_hist; i0 += svx::kMaxPartsPerLaunch) {
    const int n = std::min(svx::kMaxPartsPerLaunch, n_hist - i0);
    p.slot_base = 0;
    p.n_parts = n;
    for (int i = 0; i < n; ++i) {
      const int b = reqs[i0 + i];
      p.parts[i] = svx::PartDesc{static_cast<const __nv_bfloat16*>(k_hist_dev[b]),
                                 static_cast<const __nv_bfloat16*>(v_hist_dev[b]), 0, b,
                                 static_cast<int32_t>(hist_len_host[b])};
    }
    cudaError_t e;
    if (svx::tc_supported(head_dim, R)) {
      const int mode = svx::tc_mode_for(head_dim, n_kv_heads, R);
      int64_t slots = 0;
      const int64_t ctas = svx::tc_plan(p, mode, svx::tc_max_ctas(num_sms), &slots);
      for (int i = 0; i < n; ++i) slot_mask[p.parts[i].req] |= (1u << slots) - 1u;
      e = svx::launch_chunk_attn_tc(p, head_dim, mode, static_cast<int>(ctas), s);
    } else {
      p.n_rowblk = (R + svx::kRowsPerBlock - 1) / svx::kRowsPerBlock;
      int64_t max_tok = 0;
      for (int i = 0; i < n; ++i) max_tok = std::max<int64_t>(max_tok, p.parts[i].n_tok);
      const int64_t pairs = static_cast<int64_t>(n) * n_kv_heads * p.n_rowblk;
      int64_t sp = (2LL * num_sms + pairs - 1) / pairs;
      sp = std::min<int64_t>(sp, std::max<int64_t>(1, (max_tok + svx::kTile - 1) / svx::kTile));
      p.splits = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(sp, svx::kHistSlots)));
      for (int i = 0; i < n; ++i) {
        const int64_t nt = (static_cast<int64_t>(p.parts[i].n_tok) + svx::kTile - 1) / svx::kTile;
        for (int sp2 = 0; sp2 < p.splits; ++sp2)
          if (svx::split_tile_begin(nt, sp2 + 1, p.splits) > svx::split_tile_begin(nt, sp2, p.splits))
            slot_mask[p.parts[i].req] |= 1u << sp2;
      }
      e = svx::launch_chunk_attn(p, head_dim, s);
    }
    if (e != cudaSuccess) return fail(SVX_ERR_CUDA, "chunk kernel launch failed: %s", cudaGetErrorString(e));
  }

  // ---- candidate region, merge and finalize
  svx::FinishParams f;
  std::memset(&f, 0, sizeof(f));
  f.ws_h = ws_h;
  f.ws_a = ws_a;
  f.err = d_err;
  f.slot_stride = rows;
  f.o = static_cast<__nv_bfloat16*>(o_dev);
  f.lse = lse_dev;
  f.q = static_cast<const __nv_bfloat16*>(q_dev);
  f.k_cand = static_cast<const __nv_bfloat16*>(k_cand_dev);
  f.v_cand = static_cast<const __nv_bfloat16*>(v_cand_dev);
  f.q_scale = p.q_scale;
  f.epoch = sd.epoch;
  f.n_req = n_req;
  f.n_q_heads = n_q_heads;
  f.n_kv_heads = n_kv_heads;
  f.group = G;
  f.n_query = n_query;
  f.n_cand = n_query;
  f.tree = (k_cand_dev && parent_host) ? 1 : 0;
  if (f.tree)
    for (int i = 0; i < n_req * n_query; ++i) f.parent[i] = static_cast<int8_t>(parent_host[i]);
  for (int b = 0; b < n_req; ++b) f.slot_mask[b] = slot_mask[b];
  cudaError_t e = svx::launch_finish(f, head_dim, s);
  if (e != cudaSuccess) return fail(SVX_ERR_CUDA, "finish kernel launch failed: %s", cudaGetErrorString(e));
  return SVX_OK;
}

extern "C" svx_status svx_static_check(int32_t* expired) {
  if (!expired) return fail(SVX_ERR_INVALID_ARG, "expired is NULL");
  *expired = 0;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return fail(SVX_ERR_CUDA, "no usable current CUDA device");
  }
  StaticDevice& sd = g_devices[dev];
  std::lock_guard<std::mutex> lock(sd.mu);
  if (!sd.ready) return SVX_OK;  // no static round has run on this device
  int word = 0;
  int* d_err = reinterpret_cast<int*>(sd.ptr + kErrOffset);
  cudaError_t e = cudaDeviceSynchronize();  // every stream's static rounds have finished
  if (e == cudaSuccess) e = cudaMemcpy(&word, d_err, sizeof(int), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && word != 0) e = cudaMemset(d_err, 0, sizeof(int));
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return fail(SVX_ERR_CUDA, "static error word: %s", cudaGetErrorString(e));
  *expired = word != 0 ? 1 : 0;
  return SVX_OK;
}
