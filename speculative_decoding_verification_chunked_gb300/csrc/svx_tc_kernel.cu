// Chunk attention on the 5th-generation tensor cores (tcgen05, TMEM), d = 128.
//
// One history chunk of "Resource-Efficient Speculative Decoding for
// Long-Context LLM Serving", section 4.2, is shared by every verification query
// of the round: for a (request, KV head) pair the G*nq query rows attend to all
// tokens of the chunk, and the chunk-local online-softmax state (Eq. 7) is
// merged into the running state (Eq. 8).
//
// Shape of the work.  A KV tile of 128 tokens sits on the MMA M dimension and
// the (padded) query rows on N, so a small query group (20-64 rows) does not
// waste a 128-row MMA:
//   S^T  = K_tile . Q^T      M = 128 tokens, N = NCOL rows, K = d      (TMEM)
//   P^T  = 2^(S^T*scale - m) per row, written bf16 to shared memory
//   O^T  = V_tile^T . P^T    M = d = 128,    N = NCOL rows, K = 128 tokens (TMEM)
// and the fp32 output accumulator lives in registers (thread = one of the 128
// output dimensions), updated one tile behind the MMAs: acc = acc*alpha + O^T.
//
// Warp roles (192 threads, one CTA per SM):
//   warps 0-3  softmax and accumulation; thread t owns TMEM lane t (token t of
//              the S tile, output dimension t of the O tile)
//   warp 4     producer: 16-byte cp.async of K/V tiles into a ring of stages,
//              written in the 128-byte-swizzled layout the MMA descriptors name
//   warp 5     one thread issues the MMAs and their commits
// Work split: "stream-K" over the tiles of all (part, KV head, row block)
// pairs, so every CTA gets the same number of tiles; a CTA that covers part of
// a pair writes that segment's state into its own state slot, and the finish
// kernel merges the slots.
//
// Every mbarrier wait is bounded (2 s of global time); a wait that gives up
// raises the device error word and makes every role of the CTA stop, drain its
// copies and MMAs, free TMEM and exit.
#include <math.h>

#include "svx_internal.h"

namespace svx {
namespace {

constexpr int TOK = kTcTile;  // tokens per tile
constexpr int D = 128;
constexpr int TILE_BYTES = TOK * D * 2;  // one K or V tile, 32 KiB
constexpr int HALF_BYTES = TOK * 64 * 2; // 64 of the 128 dimensions of a tile, 16 KiB
constexpr uint64_t kWaitLimitNs = 2000000000ull;
// The running maximum of a query row (log2 units) is re-based only when a score
// exceeds it by more than kTau, so p = 2^(s - m) <= 2^kTau stays exact enough in
// bf16 and most tiles need no cross-thread maximum at all.
constexpr float kTau = 8.0f;

// Work modes of the kernel.  Every softmax warpgroup owns 32 query rows (NCOL).
//   kSingle    one warpgroup: up to 32 rows of a (request, KV head) pair per pass.
//   kRowSplit  two warpgroups on 64 rows, 32 each; both consume every K/V tile, so a tile read
//              from HBM serves all 64 rows (the token-tree shape: G = 4, 16 nodes).
enum : int { kSingle = 0, kRowSplit = 2 };

template <int MODE>
struct TcCfg {
  static constexpr int NCOL = 32;                          // query rows per warpgroup (MMA N)
  static constexpr int NWG = (MODE == kSingle) ? 1 : 2;   // softmax warpgroups
  static constexpr int ROWS = (MODE == kRowSplit) ? 2 * NCOL : NCOL;  // query rows per pass
  static constexpr int NBUF = (MODE == kRowSplit) ? 4 : 2;  // S / O / P buffers: (warpgroup, tile parity)
  static constexpr int THREADS = 32 * (4 * NWG + 2);
  static constexpr int STAGES = 3;
  static constexpr int Q_BYTES = ROWS * D * 2;
  // P^T of a tile (one per warpgroup) is written into that tile's own K buffer: K is dead once the
  // tile's S products have completed, and the stage is recycled only after its PV products.
  static constexpr int P_BYTES = NCOL * TOK * 2;
  static constexpr int OFF_KV = 0;
  static constexpr int OFF_Q = STAGES * 2 * TILE_BYTES;
  // per softmax warpgroup:
  static constexpr int OFF_RED = OFF_Q + Q_BYTES;                  // float [NWG][4][NCOL]
  static constexpr int OFF_MNEW = OFF_RED + NWG * 4 * NCOL * 4;    // float [NWG][NCOL]: reference max per row
  static constexpr int OFF_ALPHA = OFF_MNEW + NWG * NCOL * 4;      // float [NWG][2][NCOL]
  static constexpr int OFF_FIN = OFF_ALPHA + NWG * 2 * NCOL * 4;   // float [NWG][2][NCOL]: final m, l
  static constexpr int N_BAR = 2 * STAGES + 5 * NBUF + 2;
  static constexpr int OFF_BAR = OFF_FIN + NWG * 2 * NCOL * 4;
  static constexpr int OFF_MISC = OFF_BAR + N_BAR * 8;  // [0] TMEM base, [1] abort flag
  static constexpr int BYTES = OFF_MISC + 16;
  static constexpr int SMEM = BYTES + 1024;  // slack to align the base to 1024 bytes
  static constexpr uint32_t TMEM_COLS = 2 * NBUF * NCOL;  // S and O buffers: 128 or 256 columns
  static constexpr uint32_t S_COL = 0;
  static constexpr uint32_t O_COL = NBUF * NCOL;
  static_assert(OFF_Q % 1024 == 0 && P_BYTES % 1024 == 0 && (NCOL * D * 2) % 1024 == 0 &&
                    NWG * P_BYTES <= TILE_BYTES,
                "swizzle atoms need 1 KiB alignment; the P^T buffers must fit in a K tile");
  static_assert(SMEM <= 232448, "shared memory per CTA");
  // buffer of warpgroup wg for tile j
  __device__ static constexpr int buf(int64_t j, int wg) {
    return (MODE == kRowSplit) ? (wg * 2 + static_cast<int>(j & 1)) : static_cast<int>(j & 1);
  }
};

// ------------------------------------------------------------------ PTX wrappers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// Named barriers of the softmax warpgroups: id 1 + wg (its 128 threads), id 3
// (all softmax threads, at segment starts).
__device__ __forceinline__ void bar_sync(uint32_t id, uint32_t n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
// Barrier that also ANDs the threads' flags, so a wait that gave up in one
// thread makes all of them leave together.
__device__ __forceinline__ bool bar_all(uint32_t id, uint32_t n, bool ok) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.and.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(ok)), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}
// Barrier that ORs the threads' flags.
__device__ __forceinline__ bool bar_any(uint32_t id, uint32_t n, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void st_shared_b16(uint32_t addr, unsigned short v) {
  asm volatile("st.shared.b16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// 32 consecutive TMEM columns of this warp's 32 lanes into v[OFF..OFF+31]
// (thread = lane); the wait is in the same statement so no value is used early.
template <int OFF, int N>
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[N]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[OFF + i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ float exp2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Instruction descriptor of tcgen05.mma kind::f16: bf16 A and B, fp32 D.
__host__ __device__ constexpr uint32_t make_idesc(int M, int N, bool a_mn_major, bool b_mn_major) {
  return (1u << 4)                                   // D format: f32
         | (1u << 7)                                 // A format: bf16
         | (1u << 10)                                // B format: bf16
         | ((a_mn_major ? 1u : 0u) << 15)            // A major-ness
         | ((b_mn_major ? 1u : 0u) << 16)            // B major-ness
         | (static_cast<uint32_t>(N >> 3) << 17)     // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24);    // M / 16
}

// Shared-memory matrix descriptor, 128-byte swizzle (atoms of 8 rows x 128 B).
__device__ __forceinline__ uint64_t make_sdesc(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;  // descriptor version of the tcgen05 family
  d |= static_cast<uint64_t>(2) << 61;  // swizzle: 128 bytes
  return d;
}

// Byte offset of 16-byte piece `chunk` (0..15 along the 128 dimensions) of row
// `row` in a K-major, 128-byte-swizzled [rows][128] bf16 tile: two atoms
// columns of 64 dimensions, `half_bytes` apart.
__device__ __forceinline__ uint32_t swz_offset(int row, int chunk, uint32_t half_bytes) {
  return static_cast<uint32_t>(chunk >> 3) * half_bytes + static_cast<uint32_t>(row) * 128u +
         (static_cast<uint32_t>((chunk & 7) ^ (row & 7)) << 4);
}

// Butterfly transpose-reduction: on return, lane L holds the reduction over the
// warp's 32 lanes of column OFF + L (31 shuffles instead of 32 x 5).
template <int OFF, int N, bool MAX>
__device__ __forceinline__ float xpose_reduce(const float (&v)[N], int lane) {
  float w[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) w[j] = v[OFF + j];
#pragma unroll
  for (int step = 16; step >= 1; step >>= 1) {
    const bool up = (lane & step) != 0;
#pragma unroll
    for (int j = 0; j < step; ++j) {
      const float send = up ? w[j] : w[j + step];
      const float keep = up ? w[j + step] : w[j];
      const float got = __shfl_xor_sync(0xffffffffu, send, step);
      w[j] = MAX ? fmaxf(keep, got) : keep + got;
    }
  }
  return w[0];
}

struct Seg {
  int part, g, rb, slot;
  int64_t tile0;   // first tile of the segment within its part
  int64_t n_tiles;
};

// The segment of this CTA that starts at global tile x: it runs to the end of
// its (part, head, row block) pair or to the end of the CTA's range.
__device__ __forceinline__ Seg seg_at(const ChunkParams& P, int64_t x, int64_t x_end, int& hint) {
  int i = hint;
  while (i + 1 < P.n_parts && P.parts[i + 1].tile_base <= x) ++i;
  hint = i;
  const int64_t nt = (static_cast<int64_t>(P.parts[i].n_tok) + TOK - 1) / TOK;
  const int64_t local = x - P.parts[i].tile_base;
  const int64_t pair = local / nt;
  Seg s;
  s.part = i;
  s.g = static_cast<int>(pair / P.n_rowblk);
  s.rb = static_cast<int>(pair % P.n_rowblk);
  s.tile0 = local % nt;
  const int64_t first = P.parts[i].tile_base + pair * nt;
  s.n_tiles = min(x_end, first + nt) - x;
  s.slot = static_cast<int>(static_cast<int64_t>(blockIdx.x) - cta_of_tile(first, gridDim.x, P.total_tiles));
  return s;
}

struct Waiter {
  volatile uint32_t* abort;
  int* err;
  // Bounded wait that ignores the abort flag (draining in-flight MMAs).
  __device__ __forceinline__ void drain(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(bar, parity))
      if (global_ns() - t0 > kWaitLimitNs) {
        atomicOr(err, 1);
        return;
      }
  }
  // Bounded wait on an mbarrier phase; false if the CTA is aborting.
  __device__ __forceinline__ bool wait(uint32_t bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t it = 1;; ++it) {
      if (mbar_try_wait(bar, parity)) return true;
      if ((it & 255u) == 0) {
        if (*abort) return false;
        if (global_ns() - t0 > kWaitLimitNs) {
          *abort = 1u;
          atomicOr(err, 1);
          return false;
        }
      }
    }
  }
};

template <int MODE>
__global__ void __launch_bounds__(TcCfg<MODE>::THREADS, 1) chunk_attn_tc(const __grid_constant__ ChunkParams P) {
  using C = TcCfg<MODE>;
  constexpr int NCOL = C::NCOL;
  constexpr int NWG = C::NWG;
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  unsigned char* gbase = smem_raw + (base - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // mbarriers: FULL/EMPTY per stage; SFULL, SEMPTY, PFULL, OFULL, OEMPTY per buffer; QFULL; DRAIN
  const uint32_t bar0 = base + C::OFF_BAR;
  const uint32_t FULL = bar0, EMPTY = bar0 + 8u * C::STAGES;
  const uint32_t SFULL = bar0 + 16u * C::STAGES, SEMPTY = SFULL + 8u * C::NBUF, PFULL = SEMPTY + 8u * C::NBUF,
                 OFULL = PFULL + 8u * C::NBUF, OEMPTY = OFULL + 8u * C::NBUF, QFULL = OEMPTY + 8u * C::NBUF,
                 DRAIN = QFULL + 8u;
  volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(gbase + C::OFF_MISC);
  float* red = reinterpret_cast<float*>(gbase + C::OFF_RED);
  float* mnew = reinterpret_cast<float*>(gbase + C::OFF_MNEW);
  float* alpha = reinterpret_cast<float*>(gbase + C::OFF_ALPHA);
  float* fin = reinterpret_cast<float*>(gbase + C::OFF_FIN);

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(FULL + 8u * s, 32);
      mbar_init(EMPTY + 8u * s, 1);
    }
    for (int b = 0; b < C::NBUF; ++b) {
      mbar_init(SFULL + 8u * b, 1);
      mbar_init(SEMPTY + 8u * b, 128);
      mbar_init(PFULL + 8u * b, 128);
      mbar_init(OFULL + 8u * b, 1);
      mbar_init(OEMPTY + 8u * b, 128);
    }
    mbar_init(QFULL, 128 * NWG);
    mbar_init(DRAIN, 1);
    misc[1] = 0u;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    fence_proxy_async();
  }
  if (warp == 0) tmem_alloc(base + C::OFF_MISC, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  Waiter W{misc + 1, P.err};

  const int64_t T = P.total_tiles;
  const int64_t x_begin = cta_tile_begin(blockIdx.x, gridDim.x, T);
  const int64_t x_end = cta_tile_begin(blockIdx.x + 1, gridDim.x, T);
  const int64_t kv_stride = static_cast<int64_t>(P.n_kv_heads) * D;

  if (warp == 4 * NWG) {
    // ---------------- producer: K/V tiles into the stage ring
    int hint = 0;
    int64_t i = 0;
    bool ok = true;
    for (int64_t x = x_begin; x < x_end && ok;) {
      const Seg sg = seg_at(P, x, x_end, hint);
      const PartDesc& pd = P.parts[sg.part];
      const int64_t n_tok = pd.n_tok;
      const __nv_bfloat16* kb = pd.k + static_cast<int64_t>(sg.g) * D;
      const __nv_bfloat16* vb = pd.v + static_cast<int64_t>(sg.g) * D;
      for (int64_t t = 0; t < sg.n_tiles; ++t, ++i) {
        const int stage = static_cast<int>(i % C::STAGES);
        const uint32_t use = static_cast<uint32_t>(i / C::STAGES);
        if (i >= C::STAGES && !W.wait(EMPTY + 8u * stage, (use - 1u) & 1u)) {
          ok = false;
          break;
        }
        const int64_t tok0 = (sg.tile0 + t) * TOK;
        const uint32_t kdst = base + C::OFF_KV + static_cast<uint32_t>(stage) * 2u * TILE_BYTES;
        const uint32_t vdst = kdst + TILE_BYTES;
        // lane copies 16-byte piece c = lane % 16 of rows r0 + 2j (j < 64); rows past n_tok read nothing
        const int c = lane & 15, r0 = lane >> 4;
        const int64_t valid_rows = (n_tok - tok0 < TOK) ? (n_tok - tok0) : static_cast<int64_t>(TOK);
        const __nv_bfloat16* ks = kb + (tok0 + r0) * kv_stride + c * 8;
        const __nv_bfloat16* vs = vb + (tok0 + r0) * kv_stride + c * 8;
        const int64_t step = 2 * kv_stride;
        const uint32_t so0 = static_cast<uint32_t>(c >> 3) * HALF_BYTES + static_cast<uint32_t>(r0) * 128u;
#pragma unroll 8
        for (int j = 0; j < 64; ++j) {
          const int row = r0 + 2 * j;
          const uint32_t so = so0 + static_cast<uint32_t>(j) * 256u + (static_cast<uint32_t>((c & 7) ^ (row & 7)) << 4);
          const bool in = row < valid_rows;
          cp_async16(kdst + so, in ? ks : kb, in ? 16 : 0);
          cp_async16(vdst + so, in ? vs : vb, in ? 16 : 0);
          ks += step;
          vs += step;
        }
        cp_async_arrive_noinc(FULL + 8u * stage);
      }
      x += sg.n_tiles;
    }
    cp_async_wait_all();
  } else if (warp == 4 * NWG + 1) {
    // ---------------- MMA issuer (one thread)
    if (lane == 0) {
      constexpr uint32_t idesc_s = make_idesc(128, NCOL, false, false);
      constexpr uint32_t idesc_o = make_idesc(128, NCOL, true, false);
      constexpr int SGROUPS = (MODE == kRowSplit) ? 2 : 1;  // warpgroups served by one tile's MMAs
      // S^T of tile j for every warpgroup that consumes it: K tile (A, K-major) x Q rows (B, K-major)
      auto issue_s = [&](int64_t j) -> bool {
        const int stage = static_cast<int>(j % C::STAGES);
        const uint32_t use = static_cast<uint32_t>(j / C::STAGES);
        if (!W.wait(FULL + 8u * stage, use & 1u)) return false;
        fence_proxy_async();  // cp.async writes (generic proxy) before tensor-core reads (async proxy)
        const uint32_t kaddr = base + C::OFF_KV + static_cast<uint32_t>(stage) * 2u * TILE_BYTES;
        for (int g2 = 0; g2 < SGROUPS; ++g2) {
          const int wg = g2;
          const int bf = C::buf(j, wg);
          if (j >= 2 && !W.wait(SEMPTY + 8u * bf, ((static_cast<uint32_t>(j >> 1)) & 1u) ^ 1u)) return false;
          tc_fence_after();
          const uint32_t qaddr = base + C::OFF_Q + static_cast<uint32_t>((MODE == kRowSplit) ? wg : 0) * (NCOL * D * 2);
          const uint32_t d = tmem + C::S_COL + static_cast<uint32_t>(bf) * NCOL;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t a = make_sdesc(kaddr + (kk >> 2) * HALF_BYTES + (kk & 3) * 32, 16, 1024);
            const uint64_t b = make_sdesc(qaddr + (kk >> 2) * (NCOL * 128) + (kk & 3) * 32, 16, 1024);
            mma_bf16(d, a, b, idesc_s, kk > 0 ? 1u : 0u);
          }
        }
        // commits after every S product of the tile: a warpgroup writes its P^T into this K tile
        // once its SFULL fires, so no product may still be reading K then
        for (int g2 = 0; g2 < SGROUPS; ++g2)
          mma_commit(SFULL + 8u * C::buf(j, g2));
        return true;
      };
      // O^T of tile j for warpgroup wg: V tile (A, dimension-major) x P^T (B, K-major)
      auto issue_pv = [&](int64_t j, int wg) -> bool {
        const int bf = C::buf(j, wg);
        const uint32_t par = static_cast<uint32_t>(j >> 1) & 1u;
        if (!W.wait(PFULL + 8u * bf, par)) return false;
        if (j >= 2 && !W.wait(OEMPTY + 8u * bf, par ^ 1u)) return false;
        fence_proxy_async();  // P^T was written with ordinary stores
        tc_fence_after();
        const int stage = static_cast<int>(j % C::STAGES);
        const uint32_t vaddr = base + C::OFF_KV + static_cast<uint32_t>(stage) * 2u * TILE_BYTES + TILE_BYTES;
        const uint32_t paddr = base + C::OFF_KV + static_cast<uint32_t>(stage) * 2u * TILE_BYTES +
                               static_cast<uint32_t>((MODE == kRowSplit) ? wg : 0) * C::P_BYTES;
        const uint32_t d = tmem + C::O_COL + static_cast<uint32_t>(bf) * NCOL;
#pragma unroll
        for (int kk = 0; kk < TOK / 16; ++kk) {
          // A = V^T: 64-dimension halves 16 KiB apart (LBO), 8-token groups 1 KiB apart (SBO)
          const uint64_t a = make_sdesc(vaddr + kk * 2048, HALF_BYTES, 1024);
          const uint64_t b = make_sdesc(paddr + (kk >> 2) * (NCOL * 128) + (kk & 3) * 32, 16, 1024);
          mma_bf16(d, a, b, idesc_o, kk > 0 ? 1u : 0u);
        }
        mma_commit(OFULL + 8u * bf);
        return true;
      };
      int hint = 0;
      int64_t i = 0;
      uint32_t seg_idx = 0;
      bool ok = true;
      for (int64_t x = x_begin; x < x_end && ok; ++seg_idx) {
        const Seg sg = seg_at(P, x, x_end, hint);
        if (!W.wait(QFULL, seg_idx & 1u)) break;
        tc_fence_after();
        if (!issue_s(i)) break;
        for (int64_t t = 0; t < sg.n_tiles; ++t, ++i) {
          // S of the next tile goes out before this tile's PV (one tile ahead)
          if (t + 1 < sg.n_tiles && !issue_s(i + 1)) {
            ok = false;
            break;
          }
          const int stage = static_cast<int>(i % C::STAGES);
          if (MODE == kRowSplit) {
            if (!issue_pv(i, 0) || !issue_pv(i, 1)) {
              ok = false;
              break;
            }
          } else if (!issue_pv(i, 0)) {
            ok = false;
            break;
          }
          mma_commit(EMPTY + 8u * stage);  // both products of this stage are done when this fires
        }
        x += sg.n_tiles;
      }
      // drain: every MMA issued by this thread has completed before TMEM is freed
      mma_commit(DRAIN);
      W.drain(DRAIN, 0u);
    }
    __syncwarp();
  } else {
    // ---------------- softmax and accumulation: warpgroup wg = warp / 4, thread tid = TMEM lane
    // (token tid of an S tile, output dimension tid of an O tile)
    const int wg = warp >> 2;
    const int tid = threadIdx.x & 127;
    const uint32_t bar_wg = 1u + static_cast<uint32_t>(wg);
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    float acc[NCOL];  // O^T accumulator: output dimension tid, query row c
    float s[NCOL];    // scores of token tid, then p, then O^T tile values
    // Row denominators relative to mref.  One warpgroup: each thread keeps its share of every row
    // (lsum), summed once per segment.  Two warpgroups (fewer registers per thread): each tile's sums
    // are transpose-reduced at once and lane c of each warp keeps row c's partial (lw).
    constexpr bool kRowSums = (NWG == 1);
    float lsum[kRowSums ? NCOL : 1];
    float lw = 0.f;
    uint32_t rescaled = 0u;  // bit k: the tile with alpha buffer k re-based the row maxima
    float* red_w = red + wg * 4 * NCOL;
    float* mref = mnew + wg * NCOL;  // running reference maximum per row, shared by the warpgroup
    float* alpha_w = alpha + wg * 2 * NCOL;
    float* fin_w = fin + wg * 2 * NCOL;
    int hint = 0;
    int64_t i = 0;
    bool ok = true;
    int nr = NCOL;
    auto abuf = [](int64_t j) { return static_cast<int>(j & 1); };

    auto accumulate = [&](int64_t j) -> bool {
      const int bf = C::buf(j, wg);
      if (!bar_all(bar_wg, 128, W.wait(OFULL + 8u * bf, static_cast<uint32_t>(j >> 1) & 1u))) return false;
      tc_fence_after();
      tmem_ld32<0>(tmem + lane_base + C::O_COL + static_cast<uint32_t>(bf) * NCOL, s);
      tc_fence_before();
      mbar_arrive(OEMPTY + 8u * bf);
      if ((rescaled >> abuf(j)) & 1u) {
        const float4* al4 = reinterpret_cast<const float4*>(alpha_w + abuf(j) * NCOL);
#pragma unroll
        for (int c4 = 0; c4 < NCOL / 4; ++c4) {
          if (4 * c4 < nr) {
            const float4 a = al4[c4];
            acc[4 * c4 + 0] = fmaf(acc[4 * c4 + 0], a.x, s[4 * c4 + 0]);
            acc[4 * c4 + 1] = fmaf(acc[4 * c4 + 1], a.y, s[4 * c4 + 1]);
            acc[4 * c4 + 2] = fmaf(acc[4 * c4 + 2], a.z, s[4 * c4 + 2]);
            acc[4 * c4 + 3] = fmaf(acc[4 * c4 + 3], a.w, s[4 * c4 + 3]);
          }
        }
      } else {
#pragma unroll
        for (int c = 0; c < NCOL; ++c)
          if ((c & ~3) < nr) acc[c] += s[c];
      }
      return true;
    };

    for (int64_t x = x_begin; x < x_end;) {
      // all softmax threads meet here: nobody still needs the previous segment's Q, and a wait that
      // gave up anywhere stops every warpgroup together
      if (!bar_all(3u, 128u * NWG, ok)) break;
      const Seg sg = seg_at(P, x, x_end, hint);
      const PartDesc& pd = P.parts[sg.part];
      const int b = pd.req;
      const int R = P.group * P.n_query;
      const int rblk = sg.rb * C::ROWS;                          // first row of this pass
      const int nrows = min(C::ROWS, R - rblk);                   // valid rows of the pass
      const int r0 = rblk + ((MODE == kRowSplit) ? wg * NCOL : 0);  // this warpgroup's first row
      nr = max(0, min(NCOL, R - r0));
      const int64_t qrow0 =
          (static_cast<int64_t>(b) * P.n_q_heads + static_cast<int64_t>(sg.g) * P.group) * P.n_query;

      // Q rows of the pass into shared memory: 32-row K-major swizzled blocks, padding rows zero
      for (int idx = threadIdx.x; idx < C::ROWS * 16; idx += 128 * NWG) {
        const int c = idx >> 4, ch = idx & 15;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (c < nrows) v = *reinterpret_cast<const uint4*>(P.q + (qrow0 + rblk + c) * D + ch * 8);
        st_shared_v4(base + C::OFF_Q + static_cast<uint32_t>(c / NCOL) * (NCOL * D * 2) +
                         swz_offset(c % NCOL, ch, NCOL * 128),
                     v);
      }
      if ((warp & 3) == 0) mref[lane] = -INFINITY;
      fence_proxy_async();
      mbar_arrive(QFULL);

#pragma unroll
      for (int c = 0; c < NCOL; ++c) {
        acc[c] = 0.f;
        if constexpr (kRowSums) lsum[c] = 0.f;
      }
      lw = 0.f;
      int64_t prev = -1;  // this warpgroup's previous tile in the segment

      for (int64_t t = 0; t < sg.n_tiles; ++t, ++i) {
        const int bf = C::buf(i, wg);
        const bool tok_valid = (sg.tile0 + t) * TOK + tid < pd.n_tok;
        if (!bar_all(bar_wg, 128, W.wait(SFULL + 8u * bf, static_cast<uint32_t>(i >> 1) & 1u))) {
          ok = false;
          break;
        }
        tc_fence_after();
        tmem_ld32<0>(tmem + lane_base + C::S_COL + static_cast<uint32_t>(bf) * NCOL, s);
        tc_fence_before();
        mbar_arrive(SEMPTY + 8u * bf);

        // scaled scores (log2 units); does any exceed its row's reference by more than kTau?
        bool up = false;
        const float4* mr4 = reinterpret_cast<const float4*>(mref);
#pragma unroll
        for (int c4 = 0; c4 < NCOL / 4; ++c4) {
          if (4 * c4 < nr) {
            const float4 m4 = mr4[c4];
            const float mm[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int c = 4 * c4 + e;
              s[c] = tok_valid ? s[c] * P.q_scale : -INFINITY;
              up |= s[c] > mm[e] + kTau;
            }
          }
        }
        up = bar_any(bar_wg, 128, up);
        const int ab = abuf(i);
        rescaled = (rescaled & ~(1u << ab)) | (static_cast<uint32_t>(up) << ab);
        if (up) {
          // exact tile maximum per row: warp transpose-reduction, then across the 4 warps
          red_w[(warp & 3) * NCOL + lane] = xpose_reduce<0, NCOL, true>(s, lane);
          bar_sync(bar_wg, 128);
          if ((warp & 3) == 0) {
            const int c = lane;
            const float tm = fmaxf(fmaxf(red_w[c], red_w[NCOL + c]), fmaxf(red_w[2 * NCOL + c], red_w[3 * NCOL + c]));
            const float mo = mref[c];
            const float mn = fmaxf(mo, tm);
            alpha_w[ab * NCOL + c] = (mo == -INFINITY) ? 0.f : exp2_approx(mo - mn);
            mref[c] = mn;
          }
          bar_sync(bar_wg, 128);
          if constexpr (kRowSums) {
            const float4* al4 = reinterpret_cast<const float4*>(alpha_w + ab * NCOL);
#pragma unroll
            for (int c4 = 0; c4 < NCOL / 4; ++c4) {
              if (4 * c4 < nr) {
                const float4 a = al4[c4];
                lsum[4 * c4 + 0] *= a.x;
                lsum[4 * c4 + 1] *= a.y;
                lsum[4 * c4 + 2] *= a.z;
                lsum[4 * c4 + 3] *= a.w;
              }
            }
          } else {
            lw *= alpha_w[ab * NCOL + lane];
          }
        }

        // P^T = 2^(s - mref), bf16, into the K-major swizzled B operand of the PV product
        // P^T of this tile goes into the tile's K buffer (dead since the S products completed)
        const uint32_t pbase = base + C::OFF_KV + static_cast<uint32_t>(i % C::STAGES) * 2u * TILE_BYTES +
                               static_cast<uint32_t>((MODE == kRowSplit) ? wg : 0) * C::P_BYTES +
                               static_cast<uint32_t>(tid >> 6) * (NCOL * 128) + static_cast<uint32_t>((tid & 7) << 1);
#pragma unroll
        for (int c4 = 0; c4 < NCOL / 4; ++c4) {
          if (4 * c4 < nr) {
            const float4 m4 = mr4[c4];
            const float mm[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int c = 4 * c4 + e;
              const float pv = exp2_approx(s[c] - mm[e]);
              if constexpr (kRowSums) lsum[c] += pv;
              s[c] = pv;
              const uint32_t off = static_cast<uint32_t>(c) * 128u +
                                   (static_cast<uint32_t>(((tid & 63) >> 3) ^ (c & 7)) << 4);
              st_shared_b16(pbase + off, __bfloat16_as_ushort(__float2bfloat16_rn(pv)));
            }
          } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) s[4 * c4 + e] = 0.f;  // rows past nr add nothing to the sums
          }
        }
        fence_proxy_async();
        mbar_arrive(PFULL + 8u * bf);
        if constexpr (!kRowSums) lw += xpose_reduce<0, NCOL, false>(s, lane);

        // the previous tile's O one step behind, so the MMAs of tile i overlap the accumulation
        if (prev >= 0 && !accumulate(prev)) {
          ok = false;
          break;
        }
        prev = i;
      }
      if (ok && prev >= 0) ok = accumulate(prev);
      if (ok && prev >= 0) {
        // this warpgroup's segment state: m = mref, l = sum over threads, a = acc
        if constexpr (kRowSums) {
          red_w[(warp & 3) * NCOL + lane] = xpose_reduce<0, NCOL, false>(lsum, lane);
        } else {
          red_w[(warp & 3) * NCOL + lane] = lw;
        }
        bar_sync(bar_wg, 128);
        if ((warp & 3) == 0) {
          const int c = lane;
          fin_w[c] = mref[c];
          fin_w[NCOL + c] = red_w[c] + red_w[NCOL + c] + red_w[2 * NCOL + c] + red_w[3 * NCOL + c];
        }
        bar_sync(bar_wg, 128);
        const int slot = P.slot_base + sg.slot;
        const int64_t srow0 = static_cast<int64_t>(slot) * P.slot_stride + qrow0 + r0;
#pragma unroll
        for (int c = 0; c < NCOL; ++c) {
          if (c < nr) {
            const RowState old = P.ws_h[srow0 + c];
            const float m = fin_w[c];
            float a = acc[c];
            float* ap = P.ws_a + (srow0 + c) * D + tid;
            if (old.epoch == P.epoch) {
              const float mn = fmaxf(old.m, m);
              if (mn != -INFINITY) a = *ap * exp2_approx(old.m - mn) + a * exp2_approx(m - mn);
            }
            *ap = a;
          }
        }
        bar_sync(bar_wg, 128);  // every thread of the warpgroup has read the old headers (and fin)
        if (tid < nr) {
          RowState* hp = P.ws_h + srow0 + tid;
          const RowState old = *hp;
          float m = fin_w[tid], l = fin_w[NCOL + tid];
          if (old.epoch == P.epoch) {
            const float mn = fmaxf(old.m, m);
            if (mn != -INFINITY) {
              l = old.l * exp2_approx(old.m - mn) + l * exp2_approx(m - mn);
              m = mn;
            }
          }
          *hp = RowState{m, l, P.epoch, 0u};
        }
      }
      x += sg.n_tiles;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int MODE>
cudaError_t launch_tc(const ChunkParams& p, int n_ctas, cudaStream_t stream) {
  using C = TcCfg<MODE>;
  static bool configured = false;
  if (!configured) {
    cudaError_t e =
        cudaFuncSetAttribute(chunk_attn_tc<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  chunk_attn_tc<MODE><<<n_ctas, C::THREADS, C::SMEM, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

bool tc_supported(int head_dim, int rows) { return head_dim == 128 && rows >= 1; }
int tc_mode(int rows) { return rows <= TcCfg<kSingle>::ROWS ? kSingle : kRowSplit; }
int tc_rows_per_pass(int mode) { return mode == kRowSplit ? TcCfg<kRowSplit>::ROWS : TcCfg<kSingle>::ROWS; }
int tc_slots_per_segment(int) { return 1; }
int tc_max_ctas(int num_sms) { return num_sms; }  // one CTA per SM (shared memory)

cudaError_t launch_chunk_attn_tc(const ChunkParams& p, int mode, int n_ctas, cudaStream_t stream) {
  if (n_ctas < 1) return cudaSuccess;
  if (mode == kSingle) return launch_tc<kSingle>(p, n_ctas, stream);
  if (mode == kRowSplit) return launch_tc<kRowSplit>(p, n_ctas, stream);
  return cudaErrorInvalidValue;
}

}  // namespace svx
