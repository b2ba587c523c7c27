// Internal interface between the host runtime (svx_runtime.cu) and the kernels
// (svx_kernels.cu, svx_tc_kernel.cu).  Not part of the C ABI.
//
// Running state.  Each (state slot, query row) holds the online-softmax state
// of section 4.2 of "Resource-Efficient Speculative Decoding for Long-Context
// LLM Serving": m (running maximum, log2 units), l (denominator relative to m)
// and a[d] (un-normalised value sum), plus the round epoch that last wrote it.
// A kernel that finds an older epoch treats the row as empty, (-inf, 0, 0), so
// no reset pass is needed between rounds; every writer merges with Eq. (8).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace svx {

// Programmatic dependent launch.  Kernels launched with launch_pdl may start while the kernel before
// them in the stream is still running; each calls grid_dependency_wait() before its first global
// memory access (so it sees everything that kernel wrote, and what came before it in the stream) and
// allow_dependents() once the next kernel's CTAs may be scheduled: the chunk kernel when its work is
// done, the short finish kernel at once.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void allow_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename Params>
cudaError_t launch_pdl(void (*kernel)(Params), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       const Params& p) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}


// Device error word bits.  Kernels only ever set bits (atomicOr); the host reads and clears the word.
constexpr int kErrWait = 1;     // a bounded wait of the tensor-core chunk kernel gave up
constexpr int kErrExpire = 2;   // the expire-wait test hook's bounded wait ran out
constexpr int kErrBounds = 4;   // bounds-checked build: an access outside its buffer was skipped;
                                // bit 8 + site names where (BoundsSite)

// Bounds-checked build (-DSVX_BOUNDS_CHECK, libsvx_checked.so): each kernel checks that the global
// ranges it reads and writes lie in the buffers its parameters describe, and skips an access that
// does not (a load reads nothing, a store is dropped) after raising kErrBounds.  The stand-in for a
// memory checker on GPUs where none may run.  In the normal build the checks compile away.
#if defined(SVX_BOUNDS_CHECK)
constexpr bool kBoundsChecked = true;
#else
constexpr bool kBoundsChecked = false;
#endif
enum BoundsSite : int {
  kSiteTcKV = 0,    // tensor-core chunk kernel: K/V tile rows of a part
  kSiteTcQ = 1,     // tensor-core chunk kernel: Q rows
  kSiteTcState = 2, // tensor-core chunk kernel: state-slot rows
  kSiteFmaKV = 3,   // FMA chunk kernel: K/V rows
  kSiteFmaQ = 4,    // FMA chunk kernel: Q rows
  kSiteFmaState = 5,
  kSiteFinState = 6,  // finish kernel: state-slot rows
  kSiteFinIn = 7,     // finish kernel: Q and candidate K/V
  kSiteFinOut = 8,    // finish kernel: O and LSE
};

// True when [p, p + n) lies inside [base, base + extent) (element counts); in the checked build a
// false result raises kErrBounds with the site's bit.
template <typename T>
__device__ __forceinline__ bool in_bounds(const T* p, int64_t n, const T* base, int64_t extent, int* err,
                                          int site) {
  if constexpr (!kBoundsChecked) {
    return true;
  } else {
    const bool ok = base != nullptr && n >= 0 && p >= base && p + n <= base + extent;
    if (!ok) atomicOr(err, kErrBounds | (1 << (8 + site)));
    return ok;
  }
}

constexpr int kMaxReq = 256;
constexpr int kMaxPartsPerLaunch = 64;  // keeps the kernel parameter block near 2.5 KiB
constexpr int kHistSlots = 8;           // state slots per query row (history segments)
constexpr int kTile = 32;               // KV tokens per shared-memory tile (FMA kernel)
constexpr int kRowsPerBlock = 32;       // query rows (G * nq) per CTA of the FMA kernel
constexpr int kTcTile = 128;            // KV tokens per tile (tensor-core kernel, MMA M)

// Per-row state header; a[d] lives in a separate array with the same row index.
struct __align__(16) RowState {
  float m;         // running max of the scaled scores, log2 units
  float l;         // sum of 2^(s - m)
  uint32_t epoch;  // round that wrote this row
  uint32_t pad;
};

// One request's KV slice processed by one chunk-kernel launch.
struct PartDesc {
  const __nv_bfloat16* k;  // [n_tok][Hkv][d]
  const __nv_bfloat16* v;
  int64_t tile_base;  // tensor-core kernel: first tile of this part in a CTA group's tile sequence
  int32_t req;
  int32_t n_tok;
};

struct ChunkParams {
  const __nv_bfloat16* q;  // [B][Hq][nq][d]
  RowState* ws_h;          // [slots][slot_stride]
  float* ws_a;             // [slots][slot_stride][d]
  int* err;                // device error word (bounded waits that gave up, checked-build bounds)
  int64_t slot_stride;     // state rows per slot (max_req * Hq * max_query)
  int64_t q_rows;          // rows of q: n_req * Hq * nq (the bounds-checked build's extent of q)
  int64_t total_tiles;     // tensor-core kernel: tiles of one CTA group (all parts, one head and row block)
  float q_scale;           // softmax scale * log2(e)
  uint32_t epoch;          // this round
  int32_t n_q_heads;
  int32_t n_kv_heads;
  int32_t group;     // G = Hq / Hkv
  int32_t n_query;   // nq
  int32_t splits;    // FMA kernel: token splits per part (grid x)
  int32_t slot_base; // state slot of split / segment 0
  int32_t n_parts;
  int32_t n_rowblk;  // CTAs (FMA) or segments (tensor core) per (part, head) along the query rows
  // tensor-core kernel: the grid is n_kv_heads * n_rowblk CTA groups of ctas_per_group CTAs; group
  // (head g, row block rb) = blockIdx / ctas_per_group walks the tiles of every part for that head
  // and row block, split evenly over its CTAs
  int32_t ctas_per_group;
  PartDesc parts[kMaxPartsPerLaunch];
};

// Finish kernel: candidate region, merge and finalize.
struct FinishParams {
  RowState* ws_h;  // headers are read, then marked unwritten (epoch 0)
  const float* ws_a;
  int* err;        // device error word (checked-build bounds)
  int64_t slot_stride;
  __nv_bfloat16* o;              // [B][Hq][nq][d]
  float* lse;                    // [B][Hq][nq]
  const __nv_bfloat16* q;        // [B][Hq][nq][d]
  const __nv_bfloat16* k_cand;   // [B][n_cand][Hkv][d], or nullptr: no candidate region this round
  const __nv_bfloat16* v_cand;
  float q_scale;                 // softmax scale * log2(e)
  uint32_t epoch;
  int32_t n_req;
  int32_t n_q_heads;
  int32_t n_kv_heads;
  int32_t group;
  int32_t n_query;
  int32_t n_cand;                // == n_query
  int32_t tree;                  // 0: causal chain; 1: token tree given by parent[]
  int32_t pad0;
  uint32_t slot_mask[kMaxReq];   // per request: history state slots that may hold data this round
  int8_t parent[kMaxReq * 32];   // tree parents, request b node i at [b * n_query + i]; root -1
};

// FMA kernel: split s of a part with n_tiles tiles covers tiles [s*n/S, (s+1)*n/S).
__host__ __device__ inline int64_t split_tile_begin(int64_t n_tiles, int s, int splits) {
  return (n_tiles * s) / splits;
}

// Even split of T tiles over n CTAs (the tensor-core kernel's split inside a CTA group): CTA k owns
// tiles [k*T/n, (k+1)*T/n); the CTA holding tile x is cta_of_tile(x).
__host__ __device__ inline int64_t cta_tile_begin(int64_t k, int64_t n, int64_t T) { return (k * T) / n; }
__host__ __device__ inline int64_t cta_of_tile(int64_t x, int64_t n, int64_t T) { return ((x + 1) * n - 1) / T; }

cudaError_t launch_chunk_attn(const ChunkParams& p, int head_dim, cudaStream_t stream);
cudaError_t launch_finish(const FinishParams& p, int head_dim, cudaStream_t stream);
cudaError_t launch_expire_wait(int* err, uint64_t limit_ns, cudaStream_t stream);

// Tensor-core chunk kernel (d = 64 or 128).  Modes: 0 one softmax warpgroup (<= 32 query rows per pass),
// 2 two warpgroups on 32 rows each (<= 64 rows per pass), both reading every K/V tile once, 3 (d = 64)
// two warpgroups on two adjacent KV heads whose 64 dimensions form one 128-dimension tile row.
bool tc_supported(int head_dim, int rows);
int tc_mode(int rows);
// The mode for a launch: head pairs (mode 3) for head dimension 64, an even KV-head count and at most
// 32 rows per head, else tc_mode(rows).
int tc_mode_for(int head_dim, int n_kv_heads, int rows);
int tc_rows_per_pass(int mode);
int tc_slots_per_segment(int mode);
int tc_max_ctas(int num_sms);
// Work plan of a tensor-core launch over the parts already in p (n_tok set): sets n_rowblk, each
// part's tile_base, total_tiles and ctas_per_group for at most `cta_budget` CTAs, with no part
// spreading over more than kHistSlots state slots in its group.  Returns the grid size (CTA groups
// x CTAs per group) and the number of state slots used in *slots.
int64_t tc_plan(ChunkParams& p, int mode, int64_t cta_budget, int64_t* slots);
cudaError_t launch_chunk_attn_tc(const ChunkParams& p, int head_dim, int mode, int n_ctas, cudaStream_t stream);

}  // namespace svx
