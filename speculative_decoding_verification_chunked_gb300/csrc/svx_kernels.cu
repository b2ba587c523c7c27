// Kernels of the chunked multi-query verification attention
// ("Resource-Efficient Speculative Decoding for Long-Context LLM Serving",
// section 4.2, Eqs. (6)-(9)).
//
//   chunk_attn_fma<D>         history chunk: every query of the round attends to
//                             every token of the chunk (the chunk is shared by
//                             the whole query group, section 4.2), chunk-local
//                             state (Eq. 7) merged into the running state (Eq. 8).
//                             (FP32-FMA form, run only with SVX_FLAG_NO_TENSOR_CORES;
//                             by default the tensor-core kernel takes every chunk.)
//   finish_kernel<D>          the candidate region under its causal / token-tree
//                             mask (section 4.2, last paragraph), then the merge
//                             of all states (Eq. 8), O = a / l (Eq. 9) in bf16
//                             and LSE in fp32.
//
// Scores are kept in log2 units (Q is pre-multiplied by scale * log2 e) so the
// exponentials are exp2; LSE is converted back to natural log on output.
#include <math.h>

#include "svx_internal.h"

namespace svx {
namespace {

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, int src_bytes) {
  const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// 2^x with the hardware approximation (ex2.approx, flush-to-zero); 2^-inf = 0.
__device__ __forceinline__ float exp2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

constexpr float kNegInf = -INFINITY;

// ---------------------------------------------------------------------------
// Chunk attention, FMA form.
//
// Grid (splits, Hkv, n_parts * n_rowblk); 128 threads.  A CTA owns one
// (request, KV head) pair, up to 32 query rows r = (h - g*G)*nq + j of that
// KV head, and a contiguous range of 32-token tiles of the part.  K/V tiles are
// staged in shared memory with 16-byte cp.async (double-buffered); every tile
// serves all rows.  Warp w owns rows w, w+4, ..., lane t owns token t of the
// tile for the scores and columns [t*D/32, (t+1)*D/32) for the value sum.
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(128) chunk_attn_fma(const __grid_constant__ ChunkParams P) {
  constexpr int TILE = kTile;
  constexpr int KSTR = D + 8;  // padded K row: conflict-free 16-byte reads by 32 lanes
  constexpr int VPL = D / 32;  // value columns per lane
  constexpr int RPW = kRowsPerBlock / 4;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  float* sQ = reinterpret_cast<float*>(smem_raw);                       // [32][D]
  __nv_bfloat16* sK = reinterpret_cast<__nv_bfloat16*>(sQ + kRowsPerBlock * D);  // [2][TILE][KSTR]
  __nv_bfloat16* sV = sK + 2 * TILE * KSTR;                              // [2][TILE][D]

  const int split = blockIdx.x;
  const int g = blockIdx.y;
  const int p = blockIdx.z / P.n_rowblk;
  const int rb = blockIdx.z % P.n_rowblk;
  const PartDesc part = P.parts[p];
  const int64_t n_tok = part.n_tok;
  const int64_t n_tiles = (n_tok + TILE - 1) / TILE;
  const int64_t tile_lo = split_tile_begin(n_tiles, split, P.splits);
  const int64_t tile_hi = split_tile_begin(n_tiles, split + 1, P.splits);
  if (tile_lo >= tile_hi) return;  // empty split: its state slot is left untouched

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int R = P.group * P.n_query;
  const int r0 = rb * kRowsPerBlock;
  const int nr = min(kRowsPerBlock, R - r0);
  const int b = part.req;
  const int64_t row_base = (static_cast<int64_t>(b) * P.n_q_heads + static_cast<int64_t>(g) * P.group) * P.n_query;
  const int64_t kv_stride = static_cast<int64_t>(P.n_kv_heads) * D;  // elements between tokens

  auto load_tile = [&](int64_t tile, int buf) {
    constexpr int CPR = D / 8;  // 16-byte pieces per row
    const int64_t t0 = tile * TILE;
    for (int c = threadIdx.x; c < TILE * CPR; c += 128) {
      const int t = c / CPR, cc = c % CPR;
      const int64_t tok = t0 + t;
      int64_t off = tok * kv_stride + static_cast<int64_t>(g) * D + cc * 8;
      // (checked build) a row past the part, or a piece outside it, reads nothing
      const bool ok = tok < n_tok && in_bounds(part.k + off, 8, part.k, n_tok * kv_stride, P.err, kSiteFmaKV) &&
                      in_bounds(part.v + off, 8, part.v, n_tok * kv_stride, P.err, kSiteFmaKV);
      if (!ok) off = 0;
      cp_async16(sK + (buf * TILE + t) * KSTR + cc * 8, part.k + off, ok ? 16 : 0);
      cp_async16(sV + (buf * TILE + t) * D + cc * 8, part.v + off, ok ? 16 : 0);
    }
    cp_async_commit();
  };

  load_tile(tile_lo, 0);

  // Q rows of this CTA, pre-scaled into log2 units; rows past nr are zero.
  for (int i = threadIdx.x; i < kRowsPerBlock * D / 2; i += 128) {
    const int rr = (2 * i) / D, c = (2 * i) % D;
    float2 qv = make_float2(0.f, 0.f);
    if (rr < nr && in_bounds(P.q + (row_base + r0 + rr) * D + c, 2, P.q, P.q_rows * D, P.err, kSiteFmaQ)) {
      const uint32_t w = *reinterpret_cast<const uint32_t*>(P.q + (row_base + r0 + rr) * D + c);
      qv = make_float2(bf16_lo(w) * P.q_scale, bf16_hi(w) * P.q_scale);
    }
    *reinterpret_cast<float2*>(sQ + rr * D + c) = qv;
  }

  // rows owned by this warp: rr = warp + 4*i, i < nrw
  const int nrw = nr > warp ? (nr - warp + 3) / 4 : 0;
  float m[RPW], l[RPW], acc[RPW][VPL];
#pragma unroll
  for (int i = 0; i < RPW; ++i) {
    m[i] = kNegInf;
    l[i] = 0.f;
#pragma unroll
    for (int c = 0; c < VPL; ++c) acc[i][c] = 0.f;
  }

  for (int64_t tile = tile_lo; tile < tile_hi; ++tile) {
    const int buf = static_cast<int>((tile - tile_lo) & 1);
    if (tile + 1 < tile_hi) {
      load_tile(tile + 1, buf ^ 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();

    const __nv_bfloat16* kt = sK + buf * TILE * KSTR;
    const __nv_bfloat16* vt = sV + buf * TILE * D;
    const int64_t tok = tile * TILE + lane;

    // scores s[i] = q_i . k_lane (log2 units)
    float s[RPW];
#pragma unroll
    for (int i = 0; i < RPW; ++i) s[i] = 0.f;
    const __nv_bfloat16* krow = kt + lane * KSTR;
#pragma unroll 4
    for (int d0 = 0; d0 < D; d0 += 8) {
      const uint4 kw = *reinterpret_cast<const uint4*>(krow + d0);
      const float k0 = bf16_lo(kw.x), k1 = bf16_hi(kw.x), k2 = bf16_lo(kw.y), k3 = bf16_hi(kw.y);
      const float k4 = bf16_lo(kw.z), k5 = bf16_hi(kw.z), k6 = bf16_lo(kw.w), k7 = bf16_hi(kw.w);
#pragma unroll
      for (int i = 0; i < RPW; ++i) {
        if (i < nrw) {
          const float* qr = sQ + (warp + 4 * i) * D + d0;
          const float4 qa = *reinterpret_cast<const float4*>(qr);
          const float4 qb = *reinterpret_cast<const float4*>(qr + 4);
          float t = s[i];
          t = fmaf(qa.x, k0, t); t = fmaf(qa.y, k1, t); t = fmaf(qa.z, k2, t); t = fmaf(qa.w, k3, t);
          t = fmaf(qb.x, k4, t); t = fmaf(qb.y, k5, t); t = fmaf(qb.z, k6, t); t = fmaf(qb.w, k7, t);
          s[i] = t;
        }
      }
    }

    // online softmax update per row (Eqs. 7-8 folded into one step per tile)
    float pr[RPW];
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
      pr[i] = 0.f;
      if (i < nrw) {
        const bool valid = tok < n_tok;
        const float si = valid ? s[i] : kNegInf;
        const float mn = fmaxf(m[i], warp_max(si));
        if (mn != kNegInf) {
          const float alpha = exp2_approx(m[i] - mn);  // m = -inf -> 0
          pr[i] = valid ? exp2_approx(si - mn) : 0.f;
          l[i] = l[i] * alpha + pr[i];  // per-lane partial denominator
#pragma unroll
          for (int c = 0; c < VPL; ++c) acc[i][c] *= alpha;
          m[i] = mn;
        }
      }
    }

    // value sum: acc[i][c] += sum_t p_i(t) * v_t[lane*VPL + c]
#pragma unroll 4
    for (int t = 0; t < TILE; ++t) {
      float vf[VPL];
      if constexpr (VPL == 4) {
        const uint2 vw = *reinterpret_cast<const uint2*>(vt + t * D + lane * 4);
        vf[0] = bf16_lo(vw.x); vf[1] = bf16_hi(vw.x); vf[2] = bf16_lo(vw.y); vf[3] = bf16_hi(vw.y);
      } else {
        const uint32_t vw = *reinterpret_cast<const uint32_t*>(vt + t * D + lane * 2);
        vf[0] = bf16_lo(vw); vf[1] = bf16_hi(vw);
      }
#pragma unroll
      for (int i = 0; i < RPW; ++i) {
        if (i < nrw) {
          const float pt = __shfl_sync(0xffffffffu, pr[i], t);
#pragma unroll
          for (int c = 0; c < VPL; ++c) acc[i][c] = fmaf(pt, vf[c], acc[i][c]);
        }
      }
    }
    __syncthreads();  // the buffer is refilled by the next iteration's prefetch
  }

  // merge this CTA's state into its slot (Eq. 8); a row last written by an
  // older round counts as empty
  const int64_t slot_row0 = static_cast<int64_t>(P.slot_base + split) * P.slot_stride + row_base + r0;
#pragma unroll
  for (int i = 0; i < RPW; ++i) {
    if (i < nrw) {
      const int rr = warp + 4 * i;
      const float lt = warp_sum(l[i]);
      if (!in_bounds(P.ws_h + slot_row0 + rr, 1, P.ws_h, kHistSlots * P.slot_stride, P.err, kSiteFmaState)) continue;
      RowState* hp = P.ws_h + slot_row0 + rr;
      float* ap = P.ws_a + (slot_row0 + rr) * D + lane * VPL;
      const RowState old = *hp;
      float mo = m[i], lo = lt;
      float a[VPL];
#pragma unroll
      for (int c = 0; c < VPL; ++c) a[c] = acc[i][c];
      if (old.epoch == P.epoch) {
        const float mn = fmaxf(old.m, m[i]);
        if (mn != kNegInf) {
          const float al = exp2_approx(old.m - mn), be = exp2_approx(m[i] - mn);
          lo = old.l * al + lt * be;
#pragma unroll
          for (int c = 0; c < VPL; ++c) a[c] = ap[c] * al + a[c] * be;
          mo = mn;
        }
      }
      __syncwarp();  // every lane has read the old header before lane 0 replaces it
#pragma unroll
      for (int c = 0; c < VPL; ++c) ap[c] = a[c];
      if (lane == 0) *hp = RowState{mo, lo, P.epoch, 0u};
    }
  }
}

// ---------------------------------------------------------------------------
// Finish: one warp per query row (b, h, j).
//   1. Candidate region (section 4.2, last paragraph): the row attends to the
//      GPU-resident candidates its visibility word allows - candidates 0..j of a
//      causal chain, or j and its ancestors in a token tree - with the same
//      online-softmax update (Eqs. 7-8); lane t holds dimensions [t*D/32, ...).
//   2. Merge: that state and every history state slot written this round are
//      combined with Eq. (8).
//   3. O = a / l (Eq. 9) as bf16, LSE = (m + log2 l) * ln 2 as fp32.
// ---------------------------------------------------------------------------
// 128-thread blocks (four rows): with the prefetched states and candidates a thread needs ~165
// registers, and small blocks let three share an SM, so 1280 rows still fit in one wave.
constexpr int kFinishThreads = 128;

template <int D>
__global__ void __launch_bounds__(kFinishThreads) finish_kernel(const __grid_constant__ FinishParams P) {
  constexpr int VPL = D / 32;
  grid_dependency_wait();  // the chunk kernels' states (and every earlier write) are visible from here
  allow_dependents();
  const int64_t row = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t n_rows = static_cast<int64_t>(P.n_req) * P.n_q_heads * P.n_query;
  if (row >= n_rows) return;
  const int b = static_cast<int>(row / (static_cast<int64_t>(P.n_q_heads) * P.n_query));
  const int h = static_cast<int>((row / P.n_query) % P.n_q_heads);
  const int j = static_cast<int>(row % P.n_query);
  float m = kNegInf, l = 0.f, a[VPL];
#pragma unroll
  for (int c = 0; c < VPL; ++c) a[c] = 0.f;

  // The row's history states first: every header and accumulator load of the used slots is issued
  // here, so their latency overlaps the candidate region below (stale slots are loaded and ignored).
  const uint32_t smask = P.slot_mask[b];
  RowState hs[kHistSlots];
  float ha[kHistSlots][VPL];
#pragma unroll
  for (int s = 0; s < kHistSlots; ++s) {
    hs[s] = RowState{kNegInf, 0.f, 0u, 0u};
    if (((smask >> s) & 1u) &&
        in_bounds(P.ws_h + static_cast<int64_t>(s) * P.slot_stride + row, 1, P.ws_h, kHistSlots * P.slot_stride,
                  P.err, kSiteFinState)) {
      const int64_t idx = static_cast<int64_t>(s) * P.slot_stride + row;
      hs[s] = P.ws_h[idx];
      const float* ap = P.ws_a + idx * D + lane * VPL;
#pragma unroll
      for (int c = 0; c < VPL; ++c) ha[s][c] = ap[c];
    } else {
#pragma unroll
      for (int c = 0; c < VPL; ++c) ha[s][c] = 0.f;
    }
  }

  if (P.k_cand != nullptr) {
    uint32_t word;
    if (!P.tree) {
      word = (j == 31) ? 0xffffffffu : ((2u << j) - 1u);
    } else {
      word = 0u;
      int node = j;
      for (int step = 0; step < 32 && node >= 0; ++step) {  // j, then its ancestors up to the root
        word |= 1u << node;
        node = P.parent[b * P.n_query + node];
      }
    }
    float q[VPL];
    const __nv_bfloat16* qp = P.q + row * D + lane * VPL;
    const bool q_ok = in_bounds(qp, VPL, P.q, n_rows * D, P.err, kSiteFinIn);
#pragma unroll
    for (int c = 0; c < VPL; ++c) q[c] = q_ok ? __bfloat162float(qp[c]) * P.q_scale : 0.f;
    const int g = h / P.group;
    // visible candidates in batches of kCandBatch: all their K and V loads are issued first, so a
    // batch costs one memory round trip instead of one per candidate
    constexpr int kCandBatch = 8;
    while (word) {
      int idx[kCandBatch];
      int nb = 0;
#pragma unroll
      for (int t = 0; t < kCandBatch; ++t) {
        idx[t] = -1;
        if (word) {
          idx[t] = __ffs(word) - 1;
          word &= word - 1u;
          ++nb;
        }
      }
      float kk[kCandBatch][VPL], vv[kCandBatch][VPL];
#pragma unroll
      for (int t = 0; t < kCandBatch; ++t) {
        const int64_t kv_ext = static_cast<int64_t>(P.n_req) * P.n_cand * P.n_kv_heads * D;
        const int64_t kv = ((static_cast<int64_t>(b) * P.n_cand + max(idx[t], 0)) * P.n_kv_heads + g) * D + lane * VPL;
        if (idx[t] >= 0 && !(in_bounds(P.k_cand + kv, VPL, P.k_cand, kv_ext, P.err, kSiteFinIn) &&
                             in_bounds(P.v_cand + kv, VPL, P.v_cand, kv_ext, P.err, kSiteFinIn))) {
#pragma unroll
          for (int c = 0; c < VPL; ++c) kk[t][c] = vv[t][c] = 0.f;
        } else if (idx[t] >= 0) {
#pragma unroll
          for (int c = 0; c < VPL; ++c) {
            kk[t][c] = __bfloat162float(P.k_cand[kv + c]);
            vv[t][c] = __bfloat162float(P.v_cand[kv + c]);
          }
        }
      }
#pragma unroll
      for (int t = 0; t < kCandBatch; ++t) {
        if (t < nb) {
          float dot = 0.f;
#pragma unroll
          for (int c = 0; c < VPL; ++c) dot = fmaf(q[c], kk[t][c], dot);
          const float sc = warp_sum(dot);
          const float mn = fmaxf(m, sc);
          const float al = exp2_approx(m - mn), p = exp2_approx(sc - mn);
          l = l * al + p;
#pragma unroll
          for (int c = 0; c < VPL; ++c) a[c] = fmaf(p, vv[t][c], a[c] * al);
          m = mn;
        }
      }
    }
  }

  uint32_t used = 0u;
#pragma unroll
  for (int s = 0; s < kHistSlots; ++s) {
    if (!((smask >> s) & 1u) || hs[s].epoch != P.epoch) continue;  // slot not written for this row this round
    used |= 1u << s;
    const float mn = fmaxf(m, hs[s].m);
    if (mn == kNegInf) continue;
    const float al = exp2_approx(m - mn), be = exp2_approx(hs[s].m - mn);
#pragma unroll
    for (int c = 0; c < VPL; ++c) a[c] = a[c] * al + ha[s][c] * be;
    l = l * al + hs[s].l * be;
    m = mn;
  }
  // The row's slot states are consumed: mark them unwritten (epoch 0), so that nothing later takes
  // them for its own -- in particular a CUDA graph replay of this round, which reuses its epoch.
  __syncwarp();
  if (lane == 0) {
    while (used) {
      const int s = __ffs(used) - 1;
      used &= used - 1;
      P.ws_h[static_cast<int64_t>(s) * P.slot_stride + row].epoch = 0u;  // read above: in bounds
    }
  }
  __nv_bfloat16* op = P.o + row * D + lane * VPL;
  if (!(in_bounds(op, VPL, P.o, n_rows * D, P.err, kSiteFinOut) &&
        in_bounds(P.lse + row, 1, P.lse, n_rows, P.err, kSiteFinOut)))
    return;
  if (l > 0.f) {
    const float inv = 1.f / l;
#pragma unroll
    for (int c = 0; c < VPL; ++c) op[c] = __float2bfloat16_rn(a[c] * inv);
    if (lane == 0) P.lse[row] = (m + log2f(l)) * 0.69314718055994530942f;
  } else {
#pragma unroll
    for (int c = 0; c < VPL; ++c) op[c] = __float2bfloat16_rn(0.f);
    if (lane == 0) P.lse[row] = kNegInf;
  }
}

template <int D>
cudaError_t launch_chunk_fma(const ChunkParams& p, cudaStream_t stream) {
  constexpr size_t smem = kRowsPerBlock * D * sizeof(float) + 2 * kTile * (D + 8) * 2 + 2 * kTile * D * 2;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(chunk_attn_fma<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    configured = true;
  }
  dim3 grid(p.splits, p.n_kv_heads, p.n_parts * p.n_rowblk);
  chunk_attn_fma<D><<<grid, 128, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_chunk_attn(const ChunkParams& p, int head_dim, cudaStream_t stream) {
  if (head_dim == 128) return launch_chunk_fma<128>(p, stream);
  if (head_dim == 64) return launch_chunk_fma<64>(p, stream);
  return cudaErrorInvalidValue;
}

namespace {
// A bounded wait on an mbarrier phase that nothing completes: it runs out after limit_ns of global
// time and raises the device error word (kErrExpire), the way a chunk kernel's waits end when their
// producer never delivers.  Test hook of the failure path; one thread, no fault.
__global__ void expire_wait_kernel(int* err, uint64_t limit_ns) {
  __shared__ __align__(8) unsigned long long bar;
  if (threadIdx.x != 0) return;
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(&bar));
  asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(a) : "memory");
  uint64_t t0;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  for (;;) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(a)
        : "memory");
    if (done) return;
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    if (t - t0 > limit_ns) {
      atomicOr(err, kErrExpire);
      return;
    }
  }
}
}  // namespace

cudaError_t launch_expire_wait(int* err, uint64_t limit_ns, cudaStream_t stream) {
  expire_wait_kernel<<<1, 32, 0, stream>>>(err, limit_ns);
  return cudaGetLastError();
}

cudaError_t launch_finish(const FinishParams& p, int head_dim, cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(p.n_req) * p.n_q_heads * p.n_query;
  const int blocks = static_cast<int>((rows * 32 + kFinishThreads - 1) / kFinishThreads);
  if (blocks == 0) return cudaSuccess;
  if (head_dim == 128) return launch_pdl(finish_kernel<128>, dim3(blocks), dim3(kFinishThreads), 0, stream, p);
  if (head_dim == 64) return launch_pdl(finish_kernel<64>, dim3(blocks), dim3(kFinishThreads), 0, stream, p);
  return cudaErrorInvalidValue;
}

}  // namespace svx
