// Host runtime of the verification-attention library: the C ABI of svx.h, the
// round state machine, the cohort chunk planner, the copy engine (pinned host ->
// HBM staging slots on a copy stream, fenced by events) and kernel launches.
//
// Design source: "Resource-Efficient Speculative Decoding for Long-Context LLM
// Serving", section 4.2: the KV chunk is the unit of transfer and computation,
// staging buffers are reused once the whole query group has finished with them,
// transfers and attention run on separate streams, and a Cohort's requests are
// processed by one batched kernel with independent states.
#include <algorithm>
#include <array>
#include <chrono>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <new>
#include <string>
#include <thread>
#include <vector>

#include "svx.h"
#include "svx_internal.h"

using svx::ChunkParams;
using svx::FinishParams;
using svx::PartDesc;

namespace {

thread_local std::string g_create_error;

enum class RoundState { kIdle, kOpen };

constexpr int kCopyStreams = 4;  // the copy stream and three more (see svx_ctx_s::xs_more)
constexpr ptrdiff_t kMaxCopyPitch = ptrdiff_t(1) << 31;  // larger source strides: one copy per part

struct PushEvents {
  cudaEvent_t copy0, copy1, k0, k1;
  bool has_copy;
  bool zero_copy;  // the push's chunk kernel read host parts in place (no copy)
};

// Adaptive streaming (SVX_FLAG_ADAPTIVE): the context measures both transfer engines on its own pushes
// and uses the faster one.
constexpr int kRateRing = 4096;      // pushes whose transfer time is still to be read
// Per-sample decay of the time and byte sums: ~500 pushes, a whole multi-layer step.  The copy engine's
// rate can differ from one host buffer (layer) to the next; a memory of a few layers made the choice
// follow single layers and flip back and forth.
constexpr double kAdaptDecay = 0.998;
constexpr double kAdaptMargin = 0.10;   // in-place reads must be this much faster to replace the copy engine
constexpr double kAdaptBack = 0.05;     // and the copy engine this much faster than them to come back
constexpr int64_t kExploreFirst = 8;    // rounds between two measurements of the other engine, at first
constexpr int64_t kExploreMax = 1024;   // ... doubling after each measurement up to this

struct RateSample {
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  int64_t bytes = 0;
  bool in_place = false;  // timed chunk kernel that read host parts in place; else the push's copies
};

struct RoundEvents {
  cudaEvent_t begin, f0, f1;
};

// A timing window holds at most this many rounds and pushes; a round that would pass either limit
// starts a new window.
constexpr int kWindowRounds = 4096;
constexpr int kWindowPushes = 65536;

}  // namespace

namespace svx {
// Message returned by svx_last_error(NULL) on this thread.
void set_thread_error(const char* msg) { g_create_error = msg; }
}  // namespace svx

struct svx_ctx_s {
  svx_config cfg{};
  int group = 1;
  int num_sms = 0;
  cudaStream_t cs = nullptr, xs = nullptr;
  bool own_cs = false, own_xs = false;
  // Further copy streams: a chunk's copies are spread over the copy stream and these, forked from and
  // joined back into it, so several copy engines read different host buffers at once.  On hosts whose
  // memory serves one sequential copy slowly this gains 12-37%; elsewhere it changes nothing.
  std::vector<cudaStream_t> xs_more;
  std::vector<cudaEvent_t> fork_ev;                // per staging slot
  std::vector<std::vector<cudaEvent_t>> join_ev;   // per staging slot, per further copy stream

  // staging slots: n_slots buffers of max_req parts, each part = K then V
  std::vector<__nv_bfloat16*> slot_buf;
  int64_t part_elems = 0;  // max_chunk_tokens * Hkv * d
  std::vector<cudaEvent_t> slot_ready, slot_free;
  int next_slot = 0;

  // fp32 state workspace: kHistSlots history slots, rows stamped with the round epoch that wrote them
  svx::RowState* ws_h = nullptr;
  float* ws_a = nullptr;
  int64_t slot_stride = 0;
  uint32_t epoch = 0;
  int* d_err = nullptr;   // device error word: a kernel's bounded wait gave up
  bool use_tc = false;    // chunk kernel on the tensor cores

  // candidate region of the open round: computed by the finish kernel, whose launch parameters
  // carry the tree parents, so no copy is queued behind the chunk transfers
  const __nv_bfloat16* cand_k = nullptr;
  const __nv_bfloat16* cand_v = nullptr;
  std::vector<int8_t> cand_parent;  // [n_req][n_query], empty for the causal chain
  cudaEvent_t done = nullptr;

  // round
  RoundState state = RoundState::kIdle;
  int n_req = 0, n_query = 0;
  const __nv_bfloat16* q = nullptr;
  float q_scale = 0.f;
  std::vector<int64_t> hist_len;
  std::vector<uint32_t> slot_mask;               // per request, slots holding data
  std::vector<std::array<int64_t, 3>> parts_seen;  // (req, tok_start, n_tok)
  bool cand_done = false;

  // timing (SVX_FLAG_TIMING): event pools indexed by round and by push since the timing window began
  std::vector<PushEvents> ev_push;
  std::vector<RoundEvents> ev_round;
  int n_push = 0;          // pushes recorded in the window
  int n_round = 0;         // rounds begun in the window
  int round_push0 = 0;     // first push of the open round
  bool window_restart = true;  // the next round starts a new window
  int64_t h2d_bytes = 0, dev_bytes = 0;
  int n_launch = 0, n_copies = 0;
  int64_t win_h2d = 0, win_dev = 0;
  int win_launch = 0, win_copies = 0, win_rounds_done = 0;
  svx_stats last_stats{};
  int last_round = -1, last_push0 = 0, last_push1 = 0;  // the last finished round of the window
  bool last_stats_pending = false;

  // adaptive streaming: decayed sums of transfer ms and GB of host history for each engine, whose ratio
  // is the engine's recent ms per GB (< 0: not measured)
  std::vector<RateSample> rate_ring;
  int rate_head = 0, rate_tail = 0;  // samples [tail, head) wait for their transfers to complete
  double ce_ms = 0.0, ce_gb = 0.0, ip_ms = 0.0, ip_gb = 0.0;
  double ce_ms_per_gb = -1.0, ip_ms_per_gb = -1.0;
  int ce_pending = 0, ip_pending = 0;  // samples in flight per engine
  int64_t adapt_rounds = 0;            // rounds begun under the policy
  int64_t next_explore = 1, explore_gap = kExploreFirst;
  bool prefer_ip = false;              // the engine the measurements favour
  bool round_ip = false;               // the open round reads its host parts in place
  int n_zc_push = 0;                 // pushes of the open round read in place by the adaptive policy
  // A round read in place (SVX_FLAG_ZERO_COPY, or an adaptive round read in place) launches its parts
  // when it finishes, merged per request (see flush_deferred): a chunk-by-chunk push sequence then costs
  // one launch per round, not one per chunk.
  struct DeferredPart {
    PartDesc d;
    int64_t tok_start;
  };
  std::vector<DeferredPart> deferred;
  int64_t deferred_host_bytes = 0;
  bool deferred_zero_copy = false;

  // host-side fault injection (test hooks): copy submissions counted from the arming call
  int64_t copy_seq = 0, fail_at = 0, delay_at = 0;
  int32_t delay_ms = 0;
  int64_t clip_q_rows = -1;  // the q extent the chunk launches state (< 0: the real one)

  std::string err;
};

namespace {

svx_status fail(svx_ctx ctx, svx_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  if (ctx) ctx->err = buf;
  else g_create_error = buf;
  return st;
}

#define SVX_CUDA(ctx, call)                                                                            \
  do {                                                                                                 \
    cudaError_t e_ = (call);                                                                           \
    if (e_ != cudaSuccess)                                                                             \
      return fail((ctx), SVX_ERR_CUDA, "%s failed: %s (%s:%d)", #call, cudaGetErrorString(e_), __FILE__, \
                  __LINE__);                                                                           \
  } while (0)

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Memory kind of a pointer: 0 pageable/unknown, 1 pinned host, 2 device (or managed).
int pointer_kind(const void* p) {
  cudaPointerAttributes a;
  cudaError_t e = cudaPointerGetAttributes(&a, p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  if (a.type == cudaMemoryTypeHost) return 1;
  if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) return 2;
  return 0;
}

// Visibility words of the candidate region; with validate_only, checks the tree and writes nothing.
svx_status masks_impl(int32_t n_req, int32_t n_query, const int32_t* parent, uint32_t* out, std::string* why,
                      bool validate_only = false) {
  if (n_req < 0 || n_query < 1 || n_query > 32 || (!out && !validate_only)) {
    if (why) *why = "n_req >= 0, 1 <= n_query <= 32 and out != NULL required";
    return SVX_ERR_INVALID_ARG;
  }
  for (int b = 0; b < n_req; ++b) {
    const int32_t* par = parent ? parent + static_cast<int64_t>(b) * n_query : nullptr;
    if (par) {
      if (par[0] != -1) {
        if (why) *why = "tree parent[0] must be -1 (request " + std::to_string(b) + ")";
        return SVX_ERR_INVALID_ARG;
      }
      for (int i = 1; i < n_query; ++i)
        if (par[i] < 0 || par[i] >= i) {
          if (why) *why = "tree parent[i] must lie in [0, i-1] (request " + std::to_string(b) + ")";
          return SVX_ERR_INVALID_ARG;
        }
    }
    if (validate_only) continue;
    for (int j = 0; j < n_query; ++j) {
      uint32_t w;
      if (!par) {
        w = (j == 31) ? 0xffffffffu : ((1u << (j + 1)) - 1u);
      } else {
        w = 1u << j;  // a node's word is its own bit plus its parent's word
        if (j > 0) w |= out[static_cast<int64_t>(b) * n_query + par[j]];
      }
      out[static_cast<int64_t>(b) * n_query + j] = w;
    }
  }
  return SVX_OK;
}

bool coverage_impl(int32_t n_req, const int64_t* hist_len, const std::vector<std::array<int64_t, 3>>& parts,
                   std::string* why) {
  std::vector<std::vector<std::pair<int64_t, int64_t>>> per(static_cast<size_t>(std::max(n_req, 0)));
  for (const auto& p : parts) {
    const int64_t b = p[0], t0 = p[1], n = p[2];
    if (b < 0 || b >= n_req || n <= 0 || t0 < 0 || t0 > hist_len[b] || n > hist_len[b] - t0) {
      if (why) *why = "part (req " + std::to_string(b) + ", start " + std::to_string(t0) + ", n " +
                      std::to_string(n) + ") lies outside the request's history";
      return false;
    }
    per[static_cast<size_t>(b)].push_back({t0, n});
  }
  for (int b = 0; b < n_req; ++b) {
    auto& v = per[static_cast<size_t>(b)];
    std::sort(v.begin(), v.end());
    int64_t end = 0;
    for (const auto& iv : v) {
      if (iv.first != end) {
        if (why) *why = "history of request " + std::to_string(b) + (iv.first < end ? " overlaps" : " has a gap") +
                        " at token " + std::to_string(std::min(iv.first, end));
        return false;
      }
      end = iv.first + iv.second;
    }
    if (end != hist_len[b]) {
      if (why) *why = "history of request " + std::to_string(b) + " covered up to " + std::to_string(end) + " of " +
                      std::to_string(hist_len[b]) + " tokens";
      return false;
    }
  }
  return true;
}

void destroy_all(svx_ctx c) {
  if (!c) return;
  int prev = -1;
  cudaGetDevice(&prev);
  cudaSetDevice(c->cfg.device);
  if (c->cs) cudaStreamSynchronize(c->cs);
  if (c->xs) cudaStreamSynchronize(c->xs);
  for (auto s : c->xs_more) cudaStreamSynchronize(s);
  for (auto* p : c->slot_buf) cudaFree(p);
  for (auto e : c->fork_ev)
    if (e) cudaEventDestroy(e);
  for (auto& v : c->join_ev)
    for (auto e : v) cudaEventDestroy(e);
  for (auto s : c->xs_more) cudaStreamDestroy(s);
  for (auto e : c->slot_ready)
    if (e) cudaEventDestroy(e);
  for (auto e : c->slot_free)
    if (e) cudaEventDestroy(e);
  for (auto& pe : c->ev_push) {
    cudaEventDestroy(pe.copy0); cudaEventDestroy(pe.copy1); cudaEventDestroy(pe.k0); cudaEventDestroy(pe.k1);
  }
  for (auto& re : c->ev_round) {
    cudaEventDestroy(re.begin); cudaEventDestroy(re.f0); cudaEventDestroy(re.f1);
  }
  if (c->done) cudaEventDestroy(c->done);
  for (auto& rs : c->rate_ring) {
    if (rs.e0) cudaEventDestroy(rs.e0);
    if (rs.e1) cudaEventDestroy(rs.e1);
  }
  if (c->ws_h) cudaFree(c->ws_h);
  if (c->d_err) cudaFree(c->d_err);
  if (c->ws_a) cudaFree(c->ws_a);
  if (c->own_cs && c->cs) cudaStreamDestroy(c->cs);
  if (c->own_xs && c->xs) cudaStreamDestroy(c->xs);
  if (prev >= 0) cudaSetDevice(prev);
  delete c;
}

struct DeviceGuard {
  int prev = -1;
  explicit DeviceGuard(int dev) {
    cudaGetDevice(&prev);
    if (prev != dev) cudaSetDevice(dev);
  }
  ~DeviceGuard() {
    int cur = -1;
    cudaGetDevice(&cur);
    if (prev >= 0 && cur != prev) cudaSetDevice(prev);
  }
};

cudaEvent_t make_event(bool timing) {
  cudaEvent_t e = nullptr;
  if (cudaEventCreateWithFlags(&e, timing ? cudaEventDefault : cudaEventDisableTiming) != cudaSuccess) return nullptr;
  return e;
}

// Number of token splits per part for one FMA chunk-kernel launch: enough CTAs
// for about two per SM, never more tiles than the longest part has.
int choose_splits(svx_ctx c, int n_parts, int64_t max_tok, int n_rowblk) {
  const int64_t pairs = static_cast<int64_t>(n_parts) * c->cfg.n_kv_heads * n_rowblk;
  const int64_t target = 2LL * c->num_sms;
  int64_t s = (target + pairs - 1) / pairs;
  const int64_t tiles = (max_tok + svx::kTile - 1) / svx::kTile;
  s = std::min<int64_t>(s, std::max<int64_t>(tiles, 1));
  s = std::max<int64_t>(1, std::min<int64_t>(s, svx::kHistSlots));
  return static_cast<int>(s);
}

// Largest number of CTAs that one (part, head, row block) pair spreads over
// when T tiles are split evenly over n CTAs.
uint32_t nonempty_splits(int64_t n_tok, int splits) {
  const int64_t n_tiles = (n_tok + svx::kTile - 1) / svx::kTile;
  uint32_t m = 0;
  for (int s = 0; s < splits; ++s)
    if (svx::split_tile_begin(n_tiles, s + 1, splits) > svx::split_tile_begin(n_tiles, s, splits)) m |= 1u << s;
  return m;
}

}  // namespace

extern "C" {

#if defined(SVX_BOUNDS_CHECK)
const char* svx_version(void) { return "svx 0.2.0 (sm_103a, bounds-checked)"; }
#else
const char* svx_version(void) { return "svx 0.2.0 (sm_103a)"; }
#endif

int32_t svx_abi_sizes(int64_t* out, int32_t cap) {
  const int64_t sz[] = {static_cast<int64_t>(sizeof(svx_config)),     static_cast<int64_t>(sizeof(svx_part)),
                        static_cast<int64_t>(sizeof(svx_stats)),      static_cast<int64_t>(sizeof(svx_window_summary)),
                        static_cast<int64_t>(sizeof(svx_plan_entry)), static_cast<int64_t>(sizeof(svx_tier_state)),
                        static_cast<int64_t>(sizeof(svx_sched_config)), static_cast<int64_t>(sizeof(svx_draft_instr))};
  const int32_t n = static_cast<int32_t>(sizeof(sz) / sizeof(sz[0]));
  for (int32_t i = 0; i < n && i < cap; ++i) out[i] = sz[i];
  return n;
}

const char* svx_last_error(svx_ctx ctx) { return ctx ? ctx->err.c_str() : g_create_error.c_str(); }

svx_status svx_create(const svx_config* cfg, svx_ctx* out) {
  if (!out) return fail(nullptr, SVX_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (!cfg) return fail(nullptr, SVX_ERR_INVALID_ARG, "cfg is NULL");
  const svx_config& k = *cfg;
  if (k.max_req < 1 || k.max_req > svx::kMaxReq)
    return fail(nullptr, SVX_ERR_INVALID_ARG, "max_req must be in [1, %d]", svx::kMaxReq);
  if (k.n_kv_heads < 1 || k.n_q_heads < k.n_kv_heads || k.n_q_heads % k.n_kv_heads)
    return fail(nullptr, SVX_ERR_INVALID_ARG, "n_q_heads must be a positive multiple of n_kv_heads");
  if (k.head_dim != 64 && k.head_dim != 128)
    return fail(nullptr, SVX_ERR_UNSUPPORTED, "head_dim %d not supported (64 or 128)", k.head_dim);
  if (k.max_query < 1 || k.max_query > 32)
    return fail(nullptr, SVX_ERR_INVALID_ARG, "max_query must be in [1, 32]");
  if (k.max_chunk_tokens < 1) return fail(nullptr, SVX_ERR_INVALID_ARG, "max_chunk_tokens must be >= 1");
  if (k.n_slots < 2 || k.n_slots > 3) return fail(nullptr, SVX_ERR_INVALID_ARG, "n_slots must be 2 or 3");
  if (k.zero_copy_ctas < 0) return fail(nullptr, SVX_ERR_INVALID_ARG, "zero_copy_ctas must be >= 0");
  if (k.staged_ctas < 0) return fail(nullptr, SVX_ERR_INVALID_ARG, "staged_ctas must be >= 0");
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || ndev == 0) {
    cudaGetLastError();
    return fail(nullptr, SVX_ERR_CUDA, "no CUDA device available");
  }
  if (k.device < 0 || k.device >= ndev) return fail(nullptr, SVX_ERR_INVALID_ARG, "device %d out of range", k.device);
  DeviceGuard dg(k.device);
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, k.device) != cudaSuccess)
    return fail(nullptr, SVX_ERR_CUDA, "cudaGetDeviceProperties failed");
  if (prop.major < 10) return fail(nullptr, SVX_ERR_UNSUPPORTED, "needs a Blackwell GPU (sm_103a build)");

  svx_ctx c = new (std::nothrow) svx_ctx_s();
  if (!c) return fail(nullptr, SVX_ERR_OOM, "host allocation failed");
  c->cfg = k;
  c->group = k.n_q_heads / k.n_kv_heads;
  c->num_sms = prop.multiProcessorCount;
  auto bail = [&](svx_status st, const char* msg) {
    std::string m = msg;
    destroy_all(c);
    return fail(nullptr, st, "%s", m.c_str());
  };
  int lo = 0, hi = 0;
  cudaDeviceGetStreamPriorityRange(&lo, &hi);
  if (k.compute_stream) c->cs = static_cast<cudaStream_t>(k.compute_stream);
  else if (cudaStreamCreateWithPriority(&c->cs, cudaStreamNonBlocking, hi) == cudaSuccess) c->own_cs = true;
  else return bail(SVX_ERR_CUDA, "compute stream creation failed");
  if (k.copy_stream) c->xs = static_cast<cudaStream_t>(k.copy_stream);
  else if (cudaStreamCreateWithPriority(&c->xs, cudaStreamNonBlocking, hi) == cudaSuccess) c->own_xs = true;
  else return bail(SVX_ERR_CUDA, "copy stream creation failed");
  for (int i = 1; i < kCopyStreams; ++i) {
    cudaStream_t s = nullptr;
    if (cudaStreamCreateWithPriority(&s, cudaStreamNonBlocking, hi) != cudaSuccess)
      return bail(SVX_ERR_CUDA, "copy stream creation failed");
    c->xs_more.push_back(s);
  }

  c->part_elems = static_cast<int64_t>(k.max_chunk_tokens) * k.n_kv_heads * k.head_dim;
  for (int s = 0; s < k.n_slots; ++s) {
    void* p = nullptr;
    if (cudaMalloc(&p, static_cast<size_t>(c->part_elems) * 2 * 2 * k.max_req) != cudaSuccess) {
      cudaGetLastError();
      return bail(SVX_ERR_OOM, "staging slot allocation failed");
    }
    c->slot_buf.push_back(static_cast<__nv_bfloat16*>(p));
    // each event joins the context before it is checked, so a failure frees the ones already made
    c->slot_ready.push_back(make_event(false));
    c->slot_free.push_back(make_event(false));
    c->fork_ev.push_back(make_event(false));
    if (!c->slot_ready.back() || !c->slot_free.back() || !c->fork_ev.back())
      return bail(SVX_ERR_CUDA, "event creation failed");
    c->join_ev.emplace_back();
    for (size_t i = 0; i < c->xs_more.size(); ++i) {
      cudaEvent_t j = make_event(false);
      if (!j) return bail(SVX_ERR_CUDA, "event creation failed");
      c->join_ev.back().push_back(j);
    }
  }
  c->use_tc = !(k.flags & SVX_FLAG_NO_TENSOR_CORES) && svx::tc_supported(k.head_dim, c->group * k.max_query);
  c->slot_stride = static_cast<int64_t>(k.max_req) * k.n_q_heads * k.max_query;
  const int64_t n_state = static_cast<int64_t>(svx::kHistSlots) * c->slot_stride;
  if (cudaMalloc(reinterpret_cast<void**>(&c->ws_h), static_cast<size_t>(n_state) * sizeof(svx::RowState)) !=
          cudaSuccess ||
      cudaMalloc(reinterpret_cast<void**>(&c->ws_a), static_cast<size_t>(n_state) * k.head_dim * sizeof(float)) !=
          cudaSuccess ||
      cudaMalloc(reinterpret_cast<void**>(&c->d_err), sizeof(int)) != cudaSuccess) {
    cudaGetLastError();
    return bail(SVX_ERR_OOM, "workspace allocation failed");
  }
  // epoch 0 marks every state row as never written (rounds count from 1)
  if (cudaMemset(c->ws_h, 0, static_cast<size_t>(n_state) * sizeof(svx::RowState)) != cudaSuccess ||
      cudaMemset(c->d_err, 0, sizeof(int)) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
    cudaGetLastError();
    return bail(SVX_ERR_CUDA, "workspace initialisation failed");
  }
  c->done = make_event(false);
  if (!c->done) return bail(SVX_ERR_CUDA, "event creation failed");
  *out = c;
  return SVX_OK;
}

svx_status svx_destroy(svx_ctx ctx) {
  destroy_all(ctx);
  return SVX_OK;
}

namespace {
bool choose_round_in_place(svx_ctx c);  // adaptive streaming, below
}  // namespace

svx_status svx_round_begin(svx_ctx c, int32_t n_req, int32_t n_query, const void* q_dev, const int64_t* hist_len,
                           float scale) {
  if (!c) return SVX_ERR_INVALID_ARG;
  if (c->state != RoundState::kIdle) return fail(c, SVX_ERR_BAD_STATE, "svx_round_begin: a round is already open");
  if (n_req < 1 || n_req > c->cfg.max_req)
    return fail(c, SVX_ERR_INVALID_ARG, "n_req must be in [1, %d]", c->cfg.max_req);
  if (n_query < 1 || n_query > c->cfg.max_query)
    return fail(c, SVX_ERR_INVALID_ARG, "n_query must be in [1, %d]", c->cfg.max_query);
  if (!q_dev || !aligned16(q_dev)) return fail(c, SVX_ERR_INVALID_ARG, "q_dev must be a 16-byte aligned pointer");
  if (!hist_len) return fail(c, SVX_ERR_INVALID_ARG, "hist_len is NULL");
  if (!(scale >= 0.f) || std::isinf(scale)) return fail(c, SVX_ERR_INVALID_ARG, "scale must be finite and >= 0");
  DeviceGuard dg(c->cfg.device);
  if (pointer_kind(q_dev) != 2) return fail(c, SVX_ERR_INVALID_ARG, "q_dev is not device memory");
  for (int b = 0; b < n_req; ++b)
    if (hist_len[b] < 0) return fail(c, SVX_ERR_INVALID_ARG, "hist_len[%d] < 0", b);
  c->n_req = n_req;
  c->n_query = n_query;
  c->q = static_cast<const __nv_bfloat16*>(q_dev);
  const float sc = scale > 0.f ? scale : 1.0f / std::sqrt(static_cast<float>(c->cfg.head_dim));
  c->q_scale = sc * 1.4426950408889634f;
  c->hist_len.assign(hist_len, hist_len + n_req);
  c->slot_mask.assign(static_cast<size_t>(n_req), 0u);
  c->parts_seen.clear();
  c->cand_done = false;
  c->h2d_bytes = c->dev_bytes = 0;
  c->n_launch = c->n_copies = 0;
  c->n_zc_push = 0;
  c->deferred.clear();
  c->deferred_host_bytes = 0;
  c->deferred_zero_copy = false;
  c->round_ip = (c->cfg.flags & SVX_FLAG_ADAPTIVE) ? choose_round_in_place(c) : false;
  c->epoch = c->epoch == 0xffffffffu ? 1u : c->epoch + 1u;
  if (c->cfg.flags & SVX_FLAG_TIMING) {
    if (c->window_restart || c->n_round >= kWindowRounds || c->n_push >= kWindowPushes) {
      c->n_round = c->n_push = 0;
      c->win_h2d = c->win_dev = 0;
      c->win_launch = c->win_copies = c->win_rounds_done = 0;
      c->last_stats_pending = false;
      c->window_restart = false;
    }
    if (c->n_round >= static_cast<int>(c->ev_round.size())) {
      RoundEvents re{make_event(true), make_event(true), make_event(true)};
      if (!re.begin || !re.f0 || !re.f1) {
        for (cudaEvent_t e : {re.begin, re.f0, re.f1})
          if (e) cudaEventDestroy(e);
        return fail(c, SVX_ERR_CUDA, "event creation failed");
      }
      c->ev_round.push_back(re);
    }
    SVX_CUDA(c, cudaEventRecord(c->ev_round[static_cast<size_t>(c->n_round)].begin, c->cs));
    c->round_push0 = c->n_push;
  }
  c->state = RoundState::kOpen;
  return SVX_OK;
}

namespace {

// Launches the chunk kernel over `parts` (already resolved to device pointers),
// in batches of at most kMaxPartsPerLaunch parts, and records which state slots
// each request may now hold.
svx_status launch_parts(svx_ctx c, std::vector<PartDesc>& parts, int cta_cap) {
  const int R = c->group * c->n_query;
  for (size_t i0 = 0; i0 < parts.size(); i0 += svx::kMaxPartsPerLaunch) {
    const int n = static_cast<int>(std::min<size_t>(svx::kMaxPartsPerLaunch, parts.size() - i0));
    ChunkParams p;
    std::memset(&p, 0, sizeof(p));
    p.q = c->q;
    p.ws_h = c->ws_h;
    p.ws_a = c->ws_a;
    p.err = c->d_err;
    p.slot_stride = c->slot_stride;
    p.q_rows = static_cast<int64_t>(c->n_req) * c->cfg.n_q_heads * c->n_query;
    if (c->clip_q_rows >= 0) p.q_rows = std::min(p.q_rows, c->clip_q_rows);
    p.q_scale = c->q_scale;
    p.epoch = c->epoch;
    p.n_q_heads = c->cfg.n_q_heads;
    p.n_kv_heads = c->cfg.n_kv_heads;
    p.group = c->group;
    p.n_query = c->n_query;
    p.slot_base = 0;
    p.n_parts = n;
    for (int i = 0; i < n; ++i) p.parts[i] = parts[i0 + i];
    if (c->use_tc) {
      const int mode = svx::tc_mode_for(c->cfg.head_dim, c->cfg.n_kv_heads, R);
      int64_t budget = svx::tc_max_ctas(c->num_sms);
      if (cta_cap > 0) budget = std::min<int64_t>(budget, cta_cap);
      int64_t slots = 0;
      const int64_t ctas = svx::tc_plan(p, mode, budget, &slots);
      for (int i = 0; i < n; ++i) {
        uint32_t& used = c->slot_mask[static_cast<size_t>(p.parts[i].req)];
        used |= (slots >= 32 ? 0xffffffffu : ((1u << slots) - 1u));
      }
      SVX_CUDA(c, svx::launch_chunk_attn_tc(p, c->cfg.head_dim, mode, static_cast<int>(ctas), c->cs));
    } else {
      p.n_rowblk = (R + svx::kRowsPerBlock - 1) / svx::kRowsPerBlock;
      int64_t max_tok = 0;
      for (int i = 0; i < n; ++i) max_tok = std::max<int64_t>(max_tok, p.parts[i].n_tok);
      p.splits = choose_splits(c, n, max_tok, p.n_rowblk);
      if (cta_cap > 0) {
        const int64_t pairs = static_cast<int64_t>(n) * c->cfg.n_kv_heads * p.n_rowblk;
        p.splits = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(p.splits, cta_cap / std::max<int64_t>(1, pairs))));
      }
      for (int i = 0; i < n; ++i)
        c->slot_mask[static_cast<size_t>(p.parts[i].req)] |= nonempty_splits(p.parts[i].n_tok, p.splits);
      SVX_CUDA(c, svx::launch_chunk_attn(p, c->cfg.head_dim, c->cs));
    }
    ++c->n_launch;
  }
  return SVX_OK;
}

// Adaptive streaming: reads the transfer times of pushes whose transfers have completed (without
// waiting) into their engine's decayed sums.  The ratio of sums is the time per byte over the recent
// pushes, which weighs a slow push by its time (a per-push average of rates would not: copy rates on
// some hosts are bimodal, full speed or a tenth of it).
void harvest_rates(svx_ctx c) {
  while (c->rate_tail != c->rate_head) {
    RateSample& rs = c->rate_ring[static_cast<size_t>(c->rate_tail)];
    const cudaError_t q = cudaEventQuery(rs.e1);
    if (q == cudaErrorNotReady) break;
    float ms = 0.f;
    if (q == cudaSuccess && cudaEventElapsedTime(&ms, rs.e0, rs.e1) == cudaSuccess && ms > 0.f && rs.bytes > 0) {
      double& sm = rs.in_place ? c->ip_ms : c->ce_ms;
      double& sg = rs.in_place ? c->ip_gb : c->ce_gb;
      sm = kAdaptDecay * sm + static_cast<double>(ms);
      sg = kAdaptDecay * sg + static_cast<double>(rs.bytes) / 1e9;
      (rs.in_place ? c->ip_ms_per_gb : c->ce_ms_per_gb) = sm / sg;
    } else {
      cudaGetLastError();
    }
    (rs.in_place ? c->ip_pending : c->ce_pending) -= 1;
    c->rate_tail = (c->rate_tail + 1) % kRateRing;
  }
}

// The engine for a round's host parts (true = read in place), chosen when the round begins, so that no
// round mixes the engines (an in-place kernel ahead of staged ones on the compute stream would hold back
// their slots, and so the copy engine).  Round 0 is staged, round 1 read in place (each engine measured
// once); then the copy engine unless in-place reads were measured kAdaptMargin faster per byte (once
// preferred, until the copy engine is measured kAdaptBack faster than them: a copy engine whose pushes
// are fast or slow by turns would otherwise pull the choice back and forth), and a whole round on the
// other engine every explore_gap rounds, the gap doubling while the preference holds.
bool choose_round_in_place(svx_ctx c) {
  harvest_rates(c);
  const int64_t r = c->adapt_rounds++;
  if (r == 0) return false;
  if (r == 1) return true;
  const bool measured = c->ce_ms_per_gb >= 0.0 && c->ip_ms_per_gb >= 0.0;
  const bool pref = measured && (c->prefer_ip ? !(c->ce_ms_per_gb * (1.0 + kAdaptBack) < c->ip_ms_per_gb)
                                              : c->ip_ms_per_gb * (1.0 + kAdaptMargin) < c->ce_ms_per_gb);
  if (pref != c->prefer_ip) {  // the preference changed: measure the other engine again soon
    c->prefer_ip = pref;
    c->explore_gap = kExploreFirst;
    c->next_explore = r + kExploreFirst;
  }
  if (r >= c->next_explore) {
    c->next_explore = r + c->explore_gap;
    c->explore_gap = std::min(kExploreMax, 2 * c->explore_gap);
    return !pref;
  }
  return pref;
}

// A ring entry for the next transfer sample (the oldest is dropped when the ring is full).
RateSample* next_sample(svx_ctx c) {
  if (c->rate_ring.empty()) c->rate_ring.resize(kRateRing);
  const int next = (c->rate_head + 1) % kRateRing;
  if (next == c->rate_tail) {
    (c->rate_ring[static_cast<size_t>(c->rate_tail)].in_place ? c->ip_pending : c->ce_pending) -= 1;
    c->rate_tail = (c->rate_tail + 1) % kRateRing;
  }
  RateSample* rs = &c->rate_ring[static_cast<size_t>(c->rate_head)];
  if (!rs->e0) rs->e0 = make_event(true);
  if (!rs->e1) rs->e1 = make_event(true);
  return rs->e0 && rs->e1 ? rs : nullptr;
}

void commit_sample(svx_ctx c, RateSample* rs, int64_t bytes, bool in_place) {
  rs->bytes = bytes;
  rs->in_place = in_place;
  (in_place ? c->ip_pending : c->ce_pending) += 1;
  c->rate_head = (c->rate_head + 1) % kRateRing;
}

}  // namespace

svx_status svx_push_chunk(svx_ctx c, const svx_part* parts, int32_t n_parts) {
  if (!c) return SVX_ERR_INVALID_ARG;
  if (c->state != RoundState::kOpen) return fail(c, SVX_ERR_BAD_STATE, "svx_push_chunk: no open round");
  if (n_parts < 0 || (n_parts > 0 && !parts)) return fail(c, SVX_ERR_INVALID_ARG, "bad parts array");
  if (n_parts == 0) return SVX_OK;
  if (n_parts > c->n_req) return fail(c, SVX_ERR_INVALID_ARG, "more parts than requests in the round");
  DeviceGuard dg(c->cfg.device);
  const int64_t row_elems = static_cast<int64_t>(c->cfg.n_kv_heads) * c->cfg.head_dim;
  std::vector<char> seen(static_cast<size_t>(c->n_req), 0);
  std::vector<int> kind(static_cast<size_t>(n_parts));
  int n_host = 0;
  for (int i = 0; i < n_parts; ++i) {
    const svx_part& p = parts[i];
    if (p.req < 0 || p.req >= c->n_req) return fail(c, SVX_ERR_INVALID_ARG, "part %d: req %d out of range", i, p.req);
    if (seen[static_cast<size_t>(p.req)])
      return fail(c, SVX_ERR_INVALID_ARG, "part %d: request %d appears twice in one chunk", i, p.req);
    seen[static_cast<size_t>(p.req)] = 1;
    const int64_t C = c->hist_len[static_cast<size_t>(p.req)];
    if (p.n_tok < 1 || p.tok_start < 0 || p.tok_start > C || p.n_tok > C - p.tok_start)
      return fail(c, SVX_ERR_INVALID_ARG, "part %d: %d tokens from %lld outside history [0, %lld) of request %d", i,
                  p.n_tok, static_cast<long long>(p.tok_start), static_cast<long long>(C), p.req);
    if (!p.k || !p.v || !aligned16(p.k) || !aligned16(p.v))
      return fail(c, SVX_ERR_INVALID_ARG, "part %d: k and v must be non-NULL and 16-byte aligned", i);
    const int kk = pointer_kind(p.k), kv = pointer_kind(p.v);
    if (kk == 0 || kv == 0 || kk != kv)
      return fail(c, SVX_ERR_INVALID_ARG,
                  "part %d: k and v must both be pinned host memory or both device memory (pageable host memory "
                  "cannot be streamed)", i);
    kind[static_cast<size_t>(i)] = kk;
    if (kk == 1 && (c->cfg.flags & SVX_FLAG_ZERO_COPY)) {
      kind[static_cast<size_t>(i)] = 3;  // pinned host, read in place by the kernel
    } else if (kk == 1) {
      if (p.n_tok > c->cfg.max_chunk_tokens)
        return fail(c, SVX_ERR_INVALID_ARG, "part %d: %d tokens exceed max_chunk_tokens %d", i, p.n_tok,
                    c->cfg.max_chunk_tokens);
      ++n_host;
    }
  }
  std::vector<int> host_idx;  // parts the copy engine stages, in slot order
  for (int i = 0; i < n_parts; ++i)
    if (kind[static_cast<size_t>(i)] == 1) host_idx.push_back(i);
  const size_t row_bytes = static_cast<size_t>(row_elems) * 2;
  const bool adaptive = (c->cfg.flags & SVX_FLAG_ADAPTIVE) != 0;
  bool adaptive_ip = false;  // this push's host parts are read in place by the adaptive policy
  int64_t host_bytes = 0;
  if (adaptive && n_host > 0) {
    harvest_rates(c);
    for (int i : host_idx) host_bytes += 2 * static_cast<int64_t>(parts[i].n_tok) * static_cast<int64_t>(row_bytes);
    if (c->round_ip) {
      for (int i : host_idx) kind[static_cast<size_t>(i)] = 3;
      host_idx.clear();
      n_host = 0;
      adaptive_ip = true;
      ++c->n_zc_push;
    }
  }
  const bool timing = (c->cfg.flags & SVX_FLAG_TIMING) != 0 && c->n_push < kWindowPushes;
  if (timing && c->n_push >= static_cast<int>(c->ev_push.size())) {
    PushEvents pe{make_event(true), make_event(true), make_event(true), make_event(true), false, false};
    if (!pe.copy0 || !pe.copy1 || !pe.k0 || !pe.k1) return fail(c, SVX_ERR_CUDA, "event creation failed");
    c->ev_push.push_back(pe);
  }
  PushEvents* pe = timing ? &c->ev_push[static_cast<size_t>(c->n_push)] : nullptr;

  std::vector<PartDesc> desc(static_cast<size_t>(n_parts));
  int slot = -1;
  bool zero_copy = false;
  if (n_host > 0) {
    // copy engine: wait until the compute stream released the slot, then stage the host parts
    slot = c->next_slot;
    c->next_slot = (c->next_slot + 1) % c->cfg.n_slots;
    SVX_CUDA(c, cudaStreamWaitEvent(c->xs, c->slot_free[static_cast<size_t>(slot)], 0));
    RateSample* rs = nullptr;
    if (adaptive) {  // this push's copy time, read by a later push once the copies have completed
      rs = next_sample(c);
      if (!rs) return fail(c, SVX_ERR_CUDA, "event creation failed");
    }
    const size_t si = static_cast<size_t>(slot);
    // Host part h goes to slot position h: K at 2h * part_elems, V right after it.  When the host parts
    // have one length and their K (and V) pointers are equally strided in increasing order -- the
    // requests' rows of one batched [B][C][Hkv][d] tensor -- one 2D copy moves all K parts and one
    // all V parts (qwen3 chunks: 208 GB/s against 192 GB/s for 4 MiB copies one by one).
    const size_t dpitch = static_cast<size_t>(2 * c->part_elems) * 2;
    bool strided = host_idx.size() > 1;
    ptrdiff_t sk = 0, sv = 0;
    if (strided) {
      const svx_part& p0 = parts[host_idx[0]];
      const char* k0 = static_cast<const char*>(p0.k);
      const char* v0 = static_cast<const char*>(p0.v);
      sk = static_cast<const char*>(parts[host_idx[1]].k) - k0;
      sv = static_cast<const char*>(parts[host_idx[1]].v) - v0;
      const ptrdiff_t width = static_cast<ptrdiff_t>(p0.n_tok) * static_cast<ptrdiff_t>(row_bytes);
      strided = sk >= width && sv >= width && sk <= kMaxCopyPitch && sv <= kMaxCopyPitch;
      for (size_t h = 1; strided && h < host_idx.size(); ++h) {
        const svx_part& p = parts[host_idx[h]];
        strided = p.n_tok == p0.n_tok && static_cast<const char*>(p.k) - k0 == static_cast<ptrdiff_t>(h) * sk &&
                  static_cast<const char*>(p.v) - v0 == static_cast<ptrdiff_t>(h) * sv;
      }
    }
    // Two copies (one K and one V, 2D or of a single part) go on the copy stream alone: one stream already
    // fills the host link with large copies, and each fork/join adds commands between pushes.  More copies
    // are spread over the further streams, forked from and joined back into it.
    const bool fork = !strided && host_idx.size() > 1;
    // Right before the push's first copy is submitted (so a host-side pause before it shows as copy-stream
    // idle time, not as copy time): the copy-start events, then the fork, after which the further copy
    // streams start (after the slot is free).
    bool started = false;
    auto start_copies = [&]() -> cudaError_t {
      if (started) return cudaSuccess;
      started = true;
      cudaError_t e = cudaSuccess;
      if (pe && e == cudaSuccess) e = cudaEventRecord(pe->copy0, c->xs);
      if (rs && e == cudaSuccess) e = cudaEventRecord(rs->e0, c->xs);
      if (fork && e == cudaSuccess) e = cudaEventRecord(c->fork_ev[si], c->xs);
      for (auto s : c->xs_more)
        if (fork && e == cudaSuccess) e = cudaStreamWaitEvent(s, c->fork_ev[si], 0);
      return e;
    };
    size_t nc = 0;  // copies issued; with the fork, copy n goes to stream n % kCopyStreams
    auto copy_stream = [&]() {
      const size_t k = fork ? nc++ % kCopyStreams : 0;
      return k == 0 ? c->xs : c->xs_more[k - 1];
    };
    const int64_t h2d0 = c->h2d_bytes;
    const int copies0 = c->n_copies;
    // A copy submission that fails leaves the push unprocessed: the further streams are joined back (so
    // later pushes stay ordered after the copies already issued), no kernel is launched, the parts do not
    // count as pushed, and the round stays open for the chunk to be pushed again.
    auto abandon = [&](const char* what, cudaError_t e) -> svx_status {
      for (size_t k = 0; started && fork && k < c->xs_more.size(); ++k) {
        cudaEventRecord(c->join_ev[si][k], c->xs_more[k]);
        cudaStreamWaitEvent(c->xs, c->join_ev[si][k], 0);
      }
      c->h2d_bytes = h2d0;
      c->n_copies = copies0;
      return fail(c, SVX_ERR_CUDA, "%s failed: %s; the chunk was not processed (the round stays open)", what,
                  e == cudaSuccess ? "injected failure" : cudaGetErrorString(e));
    };
    // Every copy submission passes the test hooks first: a host-side delay, or a refusal (reported as
    // cudaSuccess with `injected` set, so that it is told apart from a refusal by the runtime).
    bool injected = false;
    auto hooks = [&]() {
      ++c->copy_seq;
      if (c->delay_at > 0 && c->copy_seq == c->delay_at) {
        c->delay_at = 0;
        std::this_thread::sleep_for(std::chrono::milliseconds(c->delay_ms));
      }
      if (c->fail_at > 0 && c->copy_seq == c->fail_at) {
        c->fail_at = 0;
        injected = true;
      }
      return !injected;
    };
    __nv_bfloat16* const slot_base = c->slot_buf[static_cast<size_t>(slot)];
    // A 2D copy reads only its rows, each a whole part inside its own pinned allocation.  When the rows
    // belong to different allocations cudaMemcpy2DAsync refuses the call (invalid value, nothing enqueued);
    // those parts are then copied one by one.
    auto copy_2d = [&](__nv_bfloat16* dst, const void* src, ptrdiff_t spitch, bool& ok) -> cudaError_t {
      if (!ok) return cudaSuccess;
      if (!hooks()) return cudaSuccess;
      const cudaError_t es = start_copies();
      if (es != cudaSuccess) return es;
      const size_t width = static_cast<size_t>(parts[host_idx[0]].n_tok) * row_bytes;
      const cudaError_t e = cudaMemcpy2DAsync(dst, dpitch, src, static_cast<size_t>(spitch), width, host_idx.size(),
                                              cudaMemcpyHostToDevice, copy_stream());
      if (e == cudaSuccess) {
        c->n_copies += 1;
        return cudaSuccess;
      }
      if (e != cudaErrorInvalidValue) return e;
      cudaGetLastError();
      ok = false;
      return cudaSuccess;
    };
    bool k2d = strided, v2d = strided;
    cudaError_t ce = copy_2d(slot_base, strided ? parts[host_idx[0]].k : nullptr, sk, k2d);
    if (ce != cudaSuccess || injected) return abandon("cudaMemcpy2DAsync", ce);
    ce = copy_2d(slot_base + c->part_elems, strided ? parts[host_idx[0]].v : nullptr, sv, v2d);
    if (ce != cudaSuccess || injected) return abandon("cudaMemcpy2DAsync", ce);
    for (size_t h = 0; h < host_idx.size(); ++h) {
      const int i = host_idx[h];
      const svx_part& p = parts[i];
      __nv_bfloat16* dk = slot_base + static_cast<int64_t>(h) * 2 * c->part_elems;
      __nv_bfloat16* dv = dk + c->part_elems;
      const size_t bytes = static_cast<size_t>(p.n_tok) * row_bytes;
      if (!k2d) {
        if (hooks()) ce = start_copies();
        if (ce == cudaSuccess && !injected) ce = cudaMemcpyAsync(dk, p.k, bytes, cudaMemcpyHostToDevice, copy_stream());
        if (ce != cudaSuccess || injected) return abandon("cudaMemcpyAsync", ce);
        c->n_copies += 1;
      }
      if (!v2d) {
        if (hooks()) ce = start_copies();
        if (ce == cudaSuccess && !injected) ce = cudaMemcpyAsync(dv, p.v, bytes, cudaMemcpyHostToDevice, copy_stream());
        if (ce != cudaSuccess || injected) return abandon("cudaMemcpyAsync", ce);
        c->n_copies += 1;
      }
      desc[static_cast<size_t>(i)] = PartDesc{dk, dv, 0, p.req, p.n_tok};
      c->h2d_bytes += 2 * static_cast<int64_t>(bytes);
    }
    // join: the copy stream waits for the further ones, then marks the slot ready
    for (size_t k = 0; fork && k < c->xs_more.size(); ++k) {
      SVX_CUDA(c, cudaEventRecord(c->join_ev[si][k], c->xs_more[k]));
      SVX_CUDA(c, cudaStreamWaitEvent(c->xs, c->join_ev[si][k], 0));
    }
    if (pe) SVX_CUDA(c, cudaEventRecord(pe->copy1, c->xs));
    if (rs) {
      SVX_CUDA(c, cudaEventRecord(rs->e1, c->xs));
      commit_sample(c, rs, c->h2d_bytes - h2d0, false);
    }
    SVX_CUDA(c, cudaEventRecord(c->slot_ready[static_cast<size_t>(slot)], c->xs));
    SVX_CUDA(c, cudaStreamWaitEvent(c->cs, c->slot_ready[static_cast<size_t>(slot)], 0));
  }
  for (int i = 0; i < n_parts; ++i) {
    const svx_part& p = parts[i];
    const int kd = kind[static_cast<size_t>(i)];
    if (kd == 2 || kd == 3) {
      desc[static_cast<size_t>(i)] = PartDesc{static_cast<const __nv_bfloat16*>(p.k),
                                              static_cast<const __nv_bfloat16*>(p.v), 0, p.req, p.n_tok};
      (kd == 2 ? c->dev_bytes : c->h2d_bytes) += 2 * static_cast<int64_t>(p.n_tok) * row_elems * 2;
      if (kd == 3) zero_copy = true;
    }
    c->parts_seen.push_back({p.req, p.tok_start, p.n_tok});
  }
  if (n_host == 0 && ((c->cfg.flags & SVX_FLAG_ZERO_COPY) || (adaptive && c->round_ip))) {
    // a round read in place (every round with SVX_FLAG_ZERO_COPY, or one the adaptive policy reads in
    // place) stages nothing: its parts wait for round_finish
    for (int i = 0; i < n_parts; ++i)
      c->deferred.push_back({desc[static_cast<size_t>(i)], parts[i].tok_start});
    c->deferred_host_bytes += host_bytes;
    c->deferred_zero_copy = c->deferred_zero_copy || zero_copy;
    return SVX_OK;
  }
  if (pe) {
    pe->has_copy = n_host > 0;
    pe->zero_copy = zero_copy;
    SVX_CUDA(c, cudaEventRecord(pe->k0, c->cs));
  }
  RateSample* ip_rs = nullptr;  // an in-place push's kernel time is its transfer time
  if (adaptive_ip) {
    ip_rs = next_sample(c);
    if (!ip_rs) return fail(c, SVX_ERR_CUDA, "event creation failed");
    SVX_CUDA(c, cudaEventRecord(ip_rs->e0, c->cs));
  }
  svx_status st = launch_parts(c, desc, zero_copy ? c->cfg.zero_copy_ctas : (n_host > 0 ? c->cfg.staged_ctas : 0));
  if (st != SVX_OK) return st;
  if (ip_rs) {
    SVX_CUDA(c, cudaEventRecord(ip_rs->e1, c->cs));
    commit_sample(c, ip_rs, host_bytes, true);
  }
  if (pe) {
    SVX_CUDA(c, cudaEventRecord(pe->k1, c->cs));
    ++c->n_push;
  }
  if (slot >= 0) SVX_CUDA(c, cudaEventRecord(c->slot_free[static_cast<size_t>(slot)], c->cs));
  return SVX_OK;
}

namespace {

// Launches the parts a round read in place deferred.  A part that continues the previous part of
// its request (next tokens, K and V right after it in memory) is merged into it, so a request pushed
// chunk by chunk from one buffer becomes one part.  A launch holds at most one part per request (two
// CTAs must not merge into the same state rows at once); a part that cannot join goes to a later launch
// of the round, stream-ordered after it.  Timed as one push; its kernel time is an in-place sample.
svx_status flush_deferred(svx_ctx c) {
  if (c->deferred.empty()) return SVX_OK;
  const int64_t row_elems = static_cast<int64_t>(c->cfg.n_kv_heads) * c->cfg.head_dim;
  std::vector<std::vector<PartDesc>> batches;
  std::vector<std::vector<int64_t>> batch_end;  // per batch: the request's part's end token, or -1
  std::vector<std::vector<int>> batch_at;       // per batch: the request's index in the batch, or -1
  for (const auto& dp : c->deferred) {
    const int b = dp.d.req;
    bool placed = false;
    for (size_t k = 0; k < batches.size() && !placed; ++k) {
      const int at = batch_at[k][static_cast<size_t>(b)];
      if (at < 0) {
        batch_at[k][static_cast<size_t>(b)] = static_cast<int>(batches[k].size());
        batches[k].push_back(dp.d);
        batch_end[k][static_cast<size_t>(b)] = dp.tok_start + dp.d.n_tok;
        placed = true;
      } else {
        PartDesc& cur = batches[k][static_cast<size_t>(at)];
        const int64_t n = cur.n_tok;
        if (batch_end[k][static_cast<size_t>(b)] == dp.tok_start && dp.d.k == cur.k + n * row_elems &&
            dp.d.v == cur.v + n * row_elems && n + dp.d.n_tok <= INT32_MAX) {
          cur.n_tok = static_cast<int32_t>(n + dp.d.n_tok);
          batch_end[k][static_cast<size_t>(b)] += dp.d.n_tok;
          placed = true;
        }
      }
    }
    if (!placed) {
      batches.emplace_back(1, dp.d);
      batch_end.emplace_back(static_cast<size_t>(c->n_req), -1);
      batch_at.emplace_back(static_cast<size_t>(c->n_req), -1);
      batch_end.back()[static_cast<size_t>(b)] = dp.tok_start + dp.d.n_tok;
      batch_at.back()[static_cast<size_t>(b)] = 0;
    }
  }
  const bool timing = (c->cfg.flags & SVX_FLAG_TIMING) != 0 && c->n_push < kWindowPushes;
  if (timing && c->n_push >= static_cast<int>(c->ev_push.size())) {
    PushEvents pe{make_event(true), make_event(true), make_event(true), make_event(true), false, false};
    if (!pe.copy0 || !pe.copy1 || !pe.k0 || !pe.k1) return fail(c, SVX_ERR_CUDA, "event creation failed");
    c->ev_push.push_back(pe);
  }
  PushEvents* pe = timing ? &c->ev_push[static_cast<size_t>(c->n_push)] : nullptr;
  if (pe) {
    pe->has_copy = false;
    pe->zero_copy = c->deferred_zero_copy;
    SVX_CUDA(c, cudaEventRecord(pe->k0, c->cs));
  }
  RateSample* rs = nullptr;
  if (c->deferred_host_bytes > 0) {
    rs = next_sample(c);
    if (!rs) return fail(c, SVX_ERR_CUDA, "event creation failed");
    SVX_CUDA(c, cudaEventRecord(rs->e0, c->cs));
  }
  for (auto& batch : batches) {
    svx_status st = launch_parts(c, batch, c->deferred_zero_copy ? c->cfg.zero_copy_ctas : 0);
    if (st != SVX_OK) return st;
  }
  if (rs) {
    SVX_CUDA(c, cudaEventRecord(rs->e1, c->cs));
    commit_sample(c, rs, c->deferred_host_bytes, true);
  }
  if (pe) {
    SVX_CUDA(c, cudaEventRecord(pe->k1, c->cs));
    ++c->n_push;
  }
  c->deferred.clear();
  c->deferred_host_bytes = 0;
  c->deferred_zero_copy = false;
  return SVX_OK;
}

}  // namespace

svx_status svx_candidate_attn(svx_ctx c, const void* k_dev, const void* v_dev, int32_t n_cand,
                              const int32_t* parent_host) {
  if (!c) return SVX_ERR_INVALID_ARG;
  if (c->state != RoundState::kOpen) return fail(c, SVX_ERR_BAD_STATE, "svx_candidate_attn: no open round");
  if (c->cand_done) return fail(c, SVX_ERR_BAD_STATE, "svx_candidate_attn: already called in this round");
  if (n_cand != c->n_query)
    return fail(c, SVX_ERR_INVALID_ARG, "n_cand (%d) must equal n_query (%d)", n_cand, c->n_query);
  if (!k_dev || !v_dev || !aligned16(k_dev) || !aligned16(v_dev))
    return fail(c, SVX_ERR_INVALID_ARG, "candidate k/v must be non-NULL and 16-byte aligned");
  DeviceGuard dg(c->cfg.device);
  if (pointer_kind(k_dev) != 2 || pointer_kind(v_dev) != 2)
    return fail(c, SVX_ERR_INVALID_ARG, "candidate k/v must be device memory (the candidate region is GPU-resident)");
  std::string why;
  if (masks_impl(c->n_req, c->n_query, parent_host, nullptr, &why, true) != SVX_OK)
    return fail(c, SVX_ERR_INVALID_ARG, "%s", why.c_str());
  // the candidate region is computed by the finish kernel; keep what it needs
  c->cand_k = static_cast<const __nv_bfloat16*>(k_dev);
  c->cand_v = static_cast<const __nv_bfloat16*>(v_dev);
  c->cand_parent.clear();
  if (parent_host)
    c->cand_parent.assign(parent_host, parent_host + static_cast<size_t>(c->n_req) * c->n_query);
  c->cand_done = true;
  return SVX_OK;
}

svx_status svx_round_finish(svx_ctx c, void* o_dev, float* lse_dev, int32_t timeout_ms) {
  if (!c) return SVX_ERR_INVALID_ARG;
  if (c->state != RoundState::kOpen) return fail(c, SVX_ERR_BAD_STATE, "svx_round_finish: no open round");
  if (!o_dev || !lse_dev || !aligned16(o_dev) || !aligned16(lse_dev))
    return fail(c, SVX_ERR_INVALID_ARG, "o_dev and lse_dev must be non-NULL and 16-byte aligned");
  if (timeout_ms < 0) return fail(c, SVX_ERR_INVALID_ARG, "timeout_ms must be >= 0");
  DeviceGuard dg(c->cfg.device);
  if (pointer_kind(o_dev) != 2 || pointer_kind(lse_dev) != 2)
    return fail(c, SVX_ERR_INVALID_ARG, "o_dev and lse_dev must be device memory");
  std::string why;
  if (!coverage_impl(c->n_req, c->hist_len.data(), c->parts_seen, &why)) {
    c->state = RoundState::kIdle;  // the round is abandoned; its enqueued work is harmless
    c->deferred.clear();           // and its deferred parts are never launched
    if (c->cfg.flags & SVX_FLAG_TIMING) c->n_push = c->round_push0;  // and it leaves the timing window
    return fail(c, SVX_ERR_INVALID_ARG, "chunk coverage check failed: %s", why.c_str());
  }
  {
    const svx_status st = flush_deferred(c);
    if (st != SVX_OK) return st;
  }
  FinishParams p;
  std::memset(&p, 0, sizeof(p));
  p.ws_h = c->ws_h;
  p.ws_a = c->ws_a;
  p.err = c->d_err;
  p.slot_stride = c->slot_stride;
  p.epoch = c->epoch;
  p.o = static_cast<__nv_bfloat16*>(o_dev);
  p.lse = lse_dev;
  p.q = c->q;
  p.k_cand = c->cand_done ? c->cand_k : nullptr;
  p.v_cand = c->cand_done ? c->cand_v : nullptr;
  p.q_scale = c->q_scale;
  p.n_req = c->n_req;
  p.n_q_heads = c->cfg.n_q_heads;
  p.n_kv_heads = c->cfg.n_kv_heads;
  p.group = c->group;
  p.n_query = c->n_query;
  p.n_cand = c->n_query;
  p.tree = c->cand_done && !c->cand_parent.empty() ? 1 : 0;
  if (p.tree)
    for (size_t i = 0; i < c->cand_parent.size(); ++i) p.parent[i] = static_cast<int8_t>(c->cand_parent[i]);
  for (int b = 0; b < c->n_req; ++b) p.slot_mask[b] = c->slot_mask[static_cast<size_t>(b)];
  const bool timing = (c->cfg.flags & SVX_FLAG_TIMING) != 0;
  c->state = RoundState::kIdle;
  c->clip_q_rows = -1;
  const RoundEvents* re = timing ? &c->ev_round[static_cast<size_t>(c->n_round)] : nullptr;
  if (re) SVX_CUDA(c, cudaEventRecord(re->f0, c->cs));
  SVX_CUDA(c, svx::launch_finish(p, c->cfg.head_dim, c->cs));
  if (re) SVX_CUDA(c, cudaEventRecord(re->f1, c->cs));
  SVX_CUDA(c, cudaEventRecord(c->done, c->cs));
  if (timing) {
    c->last_stats_pending = true;
    c->last_stats = svx_stats{};
    c->last_stats.h2d_bytes = c->h2d_bytes;
    c->last_stats.device_bytes = c->dev_bytes;
    c->last_stats.n_chunk_launches = c->n_launch;
    c->last_stats.n_copies = c->n_copies;
    c->last_round = c->n_round;
    c->last_push0 = c->round_push0;
    c->last_push1 = c->n_push;
    ++c->n_round;
    ++c->win_rounds_done;
    c->win_h2d += c->h2d_bytes;
    c->win_dev += c->dev_bytes;
    c->win_launch += c->n_launch;
    c->win_copies += c->n_copies;
  }
  if (timeout_ms > 0) {
    const auto deadline = std::chrono::steady_clock::now() + std::chrono::milliseconds(timeout_ms);
    for (;;) {
      cudaError_t e = cudaEventQuery(c->done);
      if (e == cudaSuccess) {
        int dev_err = 0;
        SVX_CUDA(c, cudaMemcpy(&dev_err, c->d_err, sizeof(int), cudaMemcpyDeviceToHost));
        if (dev_err) {  // the round's outputs are invalid; the word is cleared, so the context runs on
          SVX_CUDA(c, cudaMemset(c->d_err, 0, sizeof(int)));
          return fail(c, SVX_ERR_CUDA, "%s (device error word 0x%x)",
                      (dev_err & svx::kErrBounds) ? "a kernel skipped an access outside its buffers (checked build)"
                                                  : "a kernel gave up waiting",
                      dev_err);
        }
        break;
      }
      if (e != cudaErrorNotReady) return fail(c, SVX_ERR_CUDA, "round failed: %s", cudaGetErrorString(e));
      if (std::chrono::steady_clock::now() >= deadline)
        return fail(c, SVX_ERR_TIMEOUT, "round not complete after %d ms", timeout_ms);
      std::this_thread::sleep_for(std::chrono::microseconds(50));
    }
  }
  return SVX_OK;
}

namespace {

// Event intervals of one push, in ms from `origin` (negative for events before it: a copy stream can run
// ahead of the compute stream's round-begin event); the copy interval is {NaN, NaN} without copies.
svx_status push_intervals(svx_ctx c, cudaEvent_t origin, const PushEvents& pe, double iv[4]) {
  float a = 0.f;
  iv[0] = iv[1] = std::nan("");
  if (pe.has_copy) {
    SVX_CUDA(c, cudaEventElapsedTime(&a, origin, pe.copy0));
    iv[0] = a;
    SVX_CUDA(c, cudaEventElapsedTime(&a, origin, pe.copy1));
    iv[1] = a;
  }
  SVX_CUDA(c, cudaEventElapsedTime(&a, origin, pe.k0));
  iv[2] = a;
  SVX_CUDA(c, cudaEventElapsedTime(&a, origin, pe.k1));
  iv[3] = a;
  return SVX_OK;
}

// Overlap over pushes [p0, p1), in ms.  Transfer intervals are the staged pushes' copy intervals and
// the chunk kernels of pushes that read host memory in place (those kernels are the transfer).
struct Overlap {
  double copy_busy = 0.0;      // sum of copy intervals
  double transfer_busy = 0.0;  // length of the union of transfer intervals
  double kernel = 0.0;         // sum of chunk-kernel intervals
  double zc_kernel = 0.0;      // sum of the in-place pushes' chunk-kernel intervals
  double exposed = 0.0;        // kernel time of the other pushes outside every transfer interval
  double gaps = 0.0;           // copy-stream idle time between its first copy and its last
  int n_zc = 0;
};

svx_status overlap_of(svx_ctx c, cudaEvent_t origin, int p0, int p1, Overlap* o) {
  std::vector<std::pair<double, double>> cp, tr, kr;
  *o = Overlap{};
  for (int i = p0; i < p1; ++i) {
    const PushEvents& pe = c->ev_push[static_cast<size_t>(i)];
    double iv[4];
    svx_status st = push_intervals(c, origin, pe, iv);
    if (st != SVX_OK) return st;
    if (pe.has_copy) {
      cp.push_back({iv[0], iv[1]});
      tr.push_back({iv[0], iv[1]});
    }
    o->kernel += iv[3] - iv[2];
    if (pe.zero_copy) {
      tr.push_back({iv[2], iv[3]});
      o->zc_kernel += iv[3] - iv[2];
      ++o->n_zc;
    } else {
      kr.push_back({iv[2], iv[3]});
    }
  }
  std::sort(cp.begin(), cp.end());
  for (size_t i = 0; i < cp.size(); ++i) {
    o->copy_busy += cp[i].second - cp[i].first;
    if (i > 0) o->gaps += std::max(0.0, cp[i].first - cp[i - 1].second);
  }
  // union of the transfer intervals: sorted, merged, disjoint
  std::sort(tr.begin(), tr.end());
  std::vector<std::pair<double, double>> un;
  for (const auto& x : tr) {
    if (!un.empty() && x.first <= un.back().second) un.back().second = std::max(un.back().second, x.second);
    else un.push_back(x);
  }
  for (const auto& x : un) o->transfer_busy += x.second - x.first;
  for (const auto& k : kr) {
    double covered = 0.0;
    auto it = std::lower_bound(un.begin(), un.end(), std::make_pair(k.first, -1e300),
                               [](const std::pair<double, double>& x, const std::pair<double, double>& y) {
                                 return x.second < y.first;
                               });
    for (; it != un.end() && it->first < k.second; ++it)
      covered += std::max(0.0, std::min(k.second, it->second) - std::max(k.first, it->first));
    o->exposed += std::max(0.0, (k.second - k.first) - covered);
  }
  return SVX_OK;
}

}  // namespace

svx_status svx_round_stats(svx_ctx c, svx_stats* out) {
  if (!c || !out) return SVX_ERR_INVALID_ARG;
  if (!(c->cfg.flags & SVX_FLAG_TIMING)) return fail(c, SVX_ERR_BAD_STATE, "context created without SVX_FLAG_TIMING");
  if (!c->last_stats_pending) return fail(c, SVX_ERR_BAD_STATE, "no finished round to report");
  DeviceGuard dg(c->cfg.device);
  SVX_CUDA(c, cudaEventSynchronize(c->done));
  svx_stats s = c->last_stats;
  const RoundEvents& re = c->ev_round[static_cast<size_t>(c->last_round)];
  float ms = 0.f;
  SVX_CUDA(c, cudaEventElapsedTime(&ms, re.begin, re.f1));
  s.round_ms = ms;
  SVX_CUDA(c, cudaEventElapsedTime(&ms, re.f0, re.f1));
  s.finish_kernel_ms = ms;
  Overlap ov;
  svx_status st = overlap_of(c, re.begin, c->last_push0, c->last_push1, &ov);
  if (st != SVX_OK) return st;
  s.copy_busy_ms = ov.copy_busy;
  s.chunk_kernel_ms = ov.kernel;
  s.chunk_kernel_exposed_ms = ov.exposed;
  s.transfer_busy_ms = ov.transfer_busy;
  s.n_zero_copy_pushes = ov.n_zc;
  *out = s;
  return SVX_OK;
}

svx_status svx_window_reset(svx_ctx c) {
  if (!c) return SVX_ERR_INVALID_ARG;
  if (!(c->cfg.flags & SVX_FLAG_TIMING)) return fail(c, SVX_ERR_BAD_STATE, "context created without SVX_FLAG_TIMING");
  if (c->state == RoundState::kOpen) return fail(c, SVX_ERR_BAD_STATE, "svx_window_reset: a round is open");
  c->window_restart = true;
  return SVX_OK;
}

svx_status svx_window_stats(svx_ctx c, svx_window_summary* out) {
  if (!c || !out) return SVX_ERR_INVALID_ARG;
  if (!(c->cfg.flags & SVX_FLAG_TIMING)) return fail(c, SVX_ERR_BAD_STATE, "context created without SVX_FLAG_TIMING");
  if (c->window_restart || c->win_rounds_done == 0)
    return fail(c, SVX_ERR_BAD_STATE, "no finished round in the timing window");
  DeviceGuard dg(c->cfg.device);
  SVX_CUDA(c, cudaEventSynchronize(c->done));
  svx_window_summary w{};
  const RoundEvents& r0 = c->ev_round[0];
  const RoundEvents& r1 = c->ev_round[static_cast<size_t>(c->last_round)];
  float ms = 0.f;
  SVX_CUDA(c, cudaEventElapsedTime(&ms, r0.begin, r1.f1));
  w.window_ms = ms;
  // the copy stream may have started the window's first copies before the compute stream reached the
  // first round's begin event: the window then starts at the first copy
  for (int i = 0; i < c->last_push1; ++i)
    if (c->ev_push[static_cast<size_t>(i)].has_copy) {
      SVX_CUDA(c, cudaEventElapsedTime(&ms, r0.begin, c->ev_push[static_cast<size_t>(i)].copy0));
      if (ms < 0.f) w.window_ms -= ms;
      break;
    }
  for (int r = 0; r <= c->last_round; ++r) {
    SVX_CUDA(c, cudaEventElapsedTime(&ms, c->ev_round[static_cast<size_t>(r)].f0, c->ev_round[static_cast<size_t>(r)].f1));
    w.finish_kernel_ms += ms;
  }
  Overlap ov;
  svx_status st = overlap_of(c, r0.begin, 0, c->last_push1, &ov);
  if (st != SVX_OK) return st;
  w.copy_busy_ms = ov.copy_busy;
  w.copy_gap_ms = ov.gaps;
  w.chunk_kernel_ms = ov.kernel;
  w.chunk_kernel_exposed_ms = ov.exposed;
  w.transfer_busy_ms = ov.transfer_busy;
  w.zero_copy_kernel_ms = ov.zc_kernel;
  w.n_zero_copy_pushes = ov.n_zc;
  w.h2d_bytes = c->win_h2d;
  w.device_bytes = c->win_dev;
  w.n_rounds = c->win_rounds_done;
  w.n_pushes = c->last_push1;
  w.n_chunk_launches = c->win_launch;
  w.n_copies = c->win_copies;
  *out = w;
  return SVX_OK;
}

svx_status svx_window_intervals(svx_ctx c, double* out, int64_t cap, int64_t* n_out) {
  if (!c || !n_out || cap < 0 || (cap > 0 && !out)) return SVX_ERR_INVALID_ARG;
  if (!(c->cfg.flags & SVX_FLAG_TIMING)) return fail(c, SVX_ERR_BAD_STATE, "context created without SVX_FLAG_TIMING");
  if (c->window_restart || c->win_rounds_done == 0)
    return fail(c, SVX_ERR_BAD_STATE, "no finished round in the timing window");
  DeviceGuard dg(c->cfg.device);
  SVX_CUDA(c, cudaEventSynchronize(c->done));
  const int n = c->last_push1;
  for (int i = 0; i < n && i < cap; ++i) {
    svx_status st = push_intervals(c, c->ev_round[0].begin, c->ev_push[static_cast<size_t>(i)], out + 4 * i);
    if (st != SVX_OK) return st;
  }
  *n_out = n;
  return SVX_OK;
}

svx_status svx_plan_chunks(int32_t n_req, const int64_t* hist_len, int32_t chunk_tokens, int32_t n_slots,
                           svx_plan_entry* out, int64_t cap, int64_t* n_out) {
  if (n_req < 0 || (n_req > 0 && !hist_len) || chunk_tokens < 1 || n_slots < 1 || cap < 0 || !n_out ||
      (cap > 0 && !out))
    return SVX_ERR_INVALID_ARG;
  int64_t max_len = 0;
  for (int b = 0; b < n_req; ++b) {
    if (hist_len[b] < 0) return SVX_ERR_INVALID_ARG;
    max_len = std::max(max_len, hist_len[b]);
  }
  int64_t n = 0;
  const int64_t n_chunks = (max_len + chunk_tokens - 1) / chunk_tokens;
  for (int64_t j = 0; j < n_chunks; ++j) {
    const int64_t t0 = j * chunk_tokens;
    for (int b = 0; b < n_req; ++b) {
      if (hist_len[b] <= t0) continue;
      if (n < cap)
        out[n] = svx_plan_entry{static_cast<int32_t>(j), static_cast<int32_t>(j % n_slots), b,
                                static_cast<int32_t>(std::min<int64_t>(chunk_tokens, hist_len[b] - t0)), t0};
      ++n;
    }
  }
  *n_out = n;
  return SVX_OK;
}

svx_status svx_candidate_masks(int32_t n_req, int32_t n_query, const int32_t* parent, uint32_t* out) {
  return masks_impl(n_req, n_query, parent, out, nullptr);
}

svx_status svx_check_coverage(int32_t n_req, const int64_t* hist_len, const int64_t* parts, int64_t n_parts,
                              int32_t* ok_out) {
  if (n_req < 0 || (n_req > 0 && !hist_len) || n_parts < 0 || (n_parts > 0 && !parts) || !ok_out)
    return SVX_ERR_INVALID_ARG;
  for (int b = 0; b < n_req; ++b)
    if (hist_len[b] < 0) return SVX_ERR_INVALID_ARG;
  std::vector<std::array<int64_t, 3>> v(static_cast<size_t>(n_parts));
  for (int64_t i = 0; i < n_parts; ++i) v[static_cast<size_t>(i)] = {parts[3 * i], parts[3 * i + 1], parts[3 * i + 2]};
  *ok_out = coverage_impl(n_req, hist_len, v, nullptr) ? 1 : 0;
  return SVX_OK;
}

svx_status svx_debug_expire_wait(svx_ctx c, int32_t wait_ms) {
  if (!c || wait_ms < 1 || wait_ms > 2000) return SVX_ERR_INVALID_ARG;
  if (c->state == RoundState::kOpen) return fail(c, SVX_ERR_BAD_STATE, "svx_debug_expire_wait: a round is open");
  DeviceGuard dg(c->cfg.device);
  SVX_CUDA(c, svx::launch_expire_wait(c->d_err, static_cast<uint64_t>(wait_ms) * 1000000ull, c->cs));
  return SVX_OK;
}

svx_status svx_window_rounds(svx_ctx c, double* out, int64_t cap, int64_t* n_out) {
  if (!c || !n_out || cap < 0 || (cap > 0 && !out)) return SVX_ERR_INVALID_ARG;
  if (!(c->cfg.flags & SVX_FLAG_TIMING)) return fail(c, SVX_ERR_BAD_STATE, "context created without SVX_FLAG_TIMING");
  if (c->window_restart || c->win_rounds_done == 0)
    return fail(c, SVX_ERR_BAD_STATE, "no finished round in the timing window");
  DeviceGuard dg(c->cfg.device);
  SVX_CUDA(c, cudaEventSynchronize(c->done));
  const int n = c->last_round + 1;
  const cudaEvent_t origin = c->ev_round[0].begin;
  for (int r = 0; r < n && r < cap; ++r) {
    const RoundEvents& re = c->ev_round[static_cast<size_t>(r)];
    float ms = 0.f;
    SVX_CUDA(c, cudaEventElapsedTime(&ms, origin, re.begin));
    out[3 * r] = ms;
    SVX_CUDA(c, cudaEventElapsedTime(&ms, origin, re.f0));
    out[3 * r + 1] = ms;
    SVX_CUDA(c, cudaEventElapsedTime(&ms, origin, re.f1));
    out[3 * r + 2] = ms;
  }
  *n_out = n;
  return SVX_OK;
}

svx_status svx_adaptive_state(svx_ctx c, double* ce_ms_per_gb, double* ip_ms_per_gb, int32_t* prefer_in_place) {
  if (!c || !ce_ms_per_gb || !ip_ms_per_gb || !prefer_in_place) return SVX_ERR_INVALID_ARG;
  if (!(c->cfg.flags & SVX_FLAG_ADAPTIVE)) return fail(c, SVX_ERR_BAD_STATE, "context created without SVX_FLAG_ADAPTIVE");
  *ce_ms_per_gb = c->ce_ms_per_gb;
  *ip_ms_per_gb = c->ip_ms_per_gb;
  *prefer_in_place = c->prefer_ip ? 1 : 0;
  return SVX_OK;
}

svx_status svx_debug_fail_copy(svx_ctx c, int64_t nth) {
  if (!c || nth < 0) return SVX_ERR_INVALID_ARG;
  c->fail_at = nth > 0 ? c->copy_seq + nth : 0;
  return SVX_OK;
}

svx_status svx_debug_clip_q_rows(svx_ctx c, int64_t rows) {
  if (!c) return SVX_ERR_INVALID_ARG;
  c->clip_q_rows = rows < 0 ? -1 : rows;
  return SVX_OK;
}

svx_status svx_debug_delay_copy(svx_ctx c, int64_t nth, int32_t delay_ms) {
  if (!c || nth < 0 || delay_ms < 0 || delay_ms > 10000) return SVX_ERR_INVALID_ARG;
  c->delay_at = nth > 0 ? c->copy_seq + nth : 0;
  c->delay_ms = delay_ms;
  return SVX_OK;
}

svx_status svx_plan_tc(int32_t n_parts, const int32_t* n_tok, int32_t n_kv_heads, int32_t rows, int64_t cta_budget,
                       int64_t* grid, int32_t* n_groups, int32_t* ctas_per_group, int64_t* tiles_per_group,
                       int32_t* slots, int64_t* tile_base) {
  if (n_parts < 1 || n_parts > svx::kMaxPartsPerLaunch || !n_tok || n_kv_heads < 1 || rows < 1 || cta_budget < 1 ||
      !grid || !n_groups || !ctas_per_group || !tiles_per_group || !slots || !tile_base)
    return SVX_ERR_INVALID_ARG;
  ChunkParams p;
  std::memset(&p, 0, sizeof(p));
  p.n_kv_heads = n_kv_heads;
  p.group = rows;  // rows per KV head = group * n_query
  p.n_query = 1;
  p.n_parts = n_parts;
  for (int i = 0; i < n_parts; ++i) {
    if (n_tok[i] < 1) return SVX_ERR_INVALID_ARG;
    p.parts[i].n_tok = n_tok[i];
  }
  int64_t used = 0;
  *grid = svx::tc_plan(p, svx::tc_mode(rows), cta_budget, &used);
  if (p.total_tiles > INT32_MAX) return SVX_ERR_INVALID_ARG;
  *n_groups = static_cast<int32_t>(*grid / p.ctas_per_group);
  *ctas_per_group = p.ctas_per_group;
  *tiles_per_group = p.total_tiles;
  *slots = static_cast<int32_t>(used);
  for (int i = 0; i < n_parts; ++i) tile_base[i] = p.parts[i].tile_base;
  return SVX_OK;
}

}  // extern "C"
