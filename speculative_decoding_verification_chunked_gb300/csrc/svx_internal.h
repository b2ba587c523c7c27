// Internal interface between the host runtime (svx_runtime.cu) and the kernels
// (svx_kernels.cu).  Not part of the C ABI.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace svx {

constexpr int kMaxReq = 256;
constexpr int kMaxPartsPerLaunch = 64;  // keeps the kernel parameter block near 2 KiB
constexpr int kMaxHistSplits = 16;      // history state slots per request
constexpr int kTile = 32;               // KV tokens per shared-memory tile (FMA kernel)
constexpr int kRowsPerBlock = 32;       // query rows (G * nq) per CTA of the FMA kernel

// One request's KV slice processed by one chunk-kernel launch.
struct PartDesc {
  const __nv_bfloat16* k;  // [n_tok][Hkv][d]
  const __nv_bfloat16* v;
  int32_t req;
  int32_t n_tok;
  uint32_t init_mask;  // bit s: state slot (slot_base + s) holds nothing yet -> overwrite
  int32_t pad;
};

// Parameters of the chunk kernel (history chunks) and of its masked form
// (candidate region).
struct ChunkParams {
  const __nv_bfloat16* q;  // [B][Hq][nq][d]
  float2* ws_ml;           // [slots][slot_stride] running (m in log2 units, l)
  float* ws_a;             // [slots][slot_stride][d] running un-normalised value sum
  const uint32_t* vis;     // [B][nq] candidate visibility words (masked form only)
  int64_t slot_stride;     // state rows per slot (max_req * Hq * max_query)
  float q_scale;           // softmax scale * log2(e)
  int32_t n_q_heads;
  int32_t n_kv_heads;
  int32_t group;     // G = Hq / Hkv
  int32_t n_query;   // nq
  int32_t splits;    // token splits per part (CTAs along grid x)
  int32_t slot_base; // state slot of split 0
  int32_t n_parts;
  int32_t n_rowblk;  // CTAs per part along the query rows (ceil(G*nq / kRowsPerBlock))
  int32_t pad0;
  PartDesc parts[kMaxPartsPerLaunch];
};

struct FinishParams {
  const float2* ws_ml;
  const float* ws_a;
  int64_t slot_stride;
  __nv_bfloat16* o;  // [B][Hq][nq][d]
  float* lse;        // [B][Hq][nq]
  int32_t n_req;
  int32_t n_q_heads;
  int32_t n_query;
  int32_t pad0;
  uint32_t slot_mask[kMaxReq];  // per request: state slots that hold data
};

// Split s of a part with n_tiles tiles covers tiles [s*n/S, (s+1)*n/S).
__host__ __device__ inline int64_t split_tile_begin(int64_t n_tiles, int s, int splits) {
  return (n_tiles * s) / splits;
}

cudaError_t launch_chunk_attn(const ChunkParams& p, int head_dim, bool masked, cudaStream_t stream);
cudaError_t launch_finish(const FinishParams& p, int head_dim, cudaStream_t stream);

}  // namespace svx
