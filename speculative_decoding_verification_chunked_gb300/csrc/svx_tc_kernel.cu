// Chunk attention on the 5th-generation tensor cores (tcgen05, TMEM), d = 64 or 128.
//
// One history chunk of "Resource-Efficient Speculative Decoding for
// Long-Context LLM Serving", section 4.2, is shared by every verification query
// of the round: for a (request, KV head) pair the G*nq query rows attend to all
// tokens of the chunk, and the chunk-local online-softmax state (Eq. 7) is
// merged into the running state (Eq. 8).
//
// Shape of the work.  A KV tile of 128 tokens sits on the MMA M dimension and
// the (padded) query rows of a pass on N (32 or 64), so a small query group
// (20-64 rows) does not waste a 128-row MMA:
//   S^T  = K_tile . Q^T      M = 128 tokens, N = rows, K = d           (TMEM)
//   P^T  = 2^(S^T*scale - m) per row, written bf16 to shared memory
//   O^T  = V_tile^T . P^T    M = 128 dims,   N = rows, K = 128 tokens  (TMEM)
// and the fp32 output accumulator lives in registers (thread = one of the 128
// output dimensions), updated one tile behind the MMAs: acc = acc*alpha + O^T.
// Tiles always span 128 dimensions.  With d = 64 only their lower 64 are loaded:
// S takes d/16 MMAs over them, and the upper half of every V slot is zeroed once,
// so O^T rows 64..127 are zero and no thread keeps them.
//
// Warp roles (one CTA per SM; NWG = 1 or 2 softmax warpgroups of 32 rows each):
//   warps 0 .. 4NWG-1  softmax and accumulation: a thread holds 4 tokens x 8 rows
//                      of an S tile and one output dimension of an O tile
//   warp 4NWG          K producer, warp 4NWG+1 V producer: 16-byte cp.async of
//                      tiles into their rings, written in the 128-byte-swizzled
//                      layout the MMA descriptors name
//   warp 4NWG+2        one thread issues the MMAs and their commits, each product
//                      as soon as its inputs are ready
// Work split: one CTA group per (KV head, row block); a group's tiles (that head
// and row block of every part, part after part) are split evenly over its CTAs
// ("stream-K" inside the group), so CTA j of every group covers the same tokens
// and the heads of a request are read in step.  A CTA that covers a piece of a
// part writes that segment's state into its own state slot, and the finish
// kernel merges the slots.
//
// Launched with programmatic dependent launch: the kernel waits for the work
// before it in the stream only when it first touches global memory, and lets
// the next kernel be scheduled once its work is done.
//
// Every mbarrier wait is bounded (2 s of global time); a wait that gives up
// raises the device error word and makes every role of the CTA stop, drain its
// copies and MMAs, free TMEM and exit.
#include <math.h>

#include <algorithm>

#include "svx_internal.h"

namespace svx {
namespace {

constexpr int TOK = kTcTile;  // tokens per tile
constexpr int TILE_D = 128;                   // dimensions of a shared-memory tile (two swizzle atoms)
constexpr int TILE_BYTES = TOK * TILE_D * 2;  // one K or V tile, 32 KiB
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
//   kHeadPair  head dimension 64, up to 32 rows per KV head: one tile row is the 128 contiguous
//              dimensions of two adjacent KV heads (the history's [token][Hkv][64] row holds them side
//              by side), and warpgroup w takes the rows of head 2p + w.  Its Q rows fill only their
//              head's 64 dimensions (the other half is zero), so the 128-dimension S product is
//              block-diagonal: each row scores its own head's keys.  The PV product gives both heads'
//              values for every row, and each thread keeps the half of O that belongs to its
//              warpgroup's head.  A tile then carries 128 dimensions of history for the same softmax
//              work, as with d = 128.
enum : int { kSingle = 0, kRowSplit = 2, kHeadPair = 3 };

template <int MODE>
struct TcCfg {
  static constexpr int NCOL = 32;                          // query rows per softmax warpgroup
  static constexpr int NWG = (MODE == kSingle) ? 1 : 2;   // softmax warpgroups
  static constexpr int ROWS = NWG * NCOL;                  // query rows per pass: the MMA N of both products
  static constexpr int THREADS = 32 * (4 * NWG + 3);
  // K and V tiles sit in two rings of their own: a K slot is refilled as soon as its tile's S product
  // completes, a V slot once the PV product completes.  With one CTA per SM, 2 + 3 slots keep ~24 MB
  // of loads in flight on the whole GPU: enough for the HBM rate at its loaded latency, while a third
  // K slot (~29 MB) only lengthened DRAM queues and cost 7% (qwen3 shape, one GB300).
  static constexpr int KST = 2;  // K slots
  static constexpr int VST = 3;  // V slots
  static constexpr int Q_BYTES = ROWS * TILE_D * 2;
  static constexpr int P_BYTES = ROWS * TOK * 2;  // P^T of a tile (all rows of the pass), two buffers
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = KST * TILE_BYTES;
  static constexpr int OFF_P = OFF_V + VST * TILE_BYTES;
  static constexpr int OFF_Q = OFF_P + 2 * P_BYTES;
  // per softmax warpgroup:
  static constexpr int OFF_RED = OFF_Q + Q_BYTES;                  // float [NWG][4][NCOL]
  static constexpr int OFF_MNEW = OFF_RED + NWG * 4 * NCOL * 4;    // float [NWG][NCOL]: reference max per row
  static constexpr int OFF_ALPHA = OFF_MNEW + NWG * NCOL * 4;      // float [NWG][2][NCOL]
  static constexpr int OFF_FIN = OFF_ALPHA + NWG * 2 * NCOL * 4;   // float [NWG][2][NCOL]: final m, l
  static constexpr int N_BAR = 2 * KST + 2 * VST + 5 * 2 + 2;
  static constexpr int OFF_HDR = OFF_FIN + NWG * 2 * NCOL * 4;   // RowState [NWG][NCOL]: slot headers read back
  static constexpr int OFF_BAR = OFF_HDR + NWG * NCOL * 16;
  static constexpr int OFF_MISC = OFF_BAR + N_BAR * 8;  // [0] TMEM base, [1] abort flag
  static constexpr int BYTES = OFF_MISC + 16;
  static constexpr int SMEM = BYTES + 1024;  // slack to align the base to 1024 bytes
  // TMEM: S and O accumulators for two tile parities, ROWS columns each (128 or 256 columns); the
  // columns of warpgroup wg start at wg * NCOL within each
  static constexpr uint32_t TMEM_COLS = 4 * ROWS;
  static constexpr uint32_t S_COL = 0;
  static constexpr uint32_t O_COL = 2 * ROWS;
  static_assert(OFF_Q % 1024 == 0 && P_BYTES % 1024 == 0 && Q_BYTES % 1024 == 0,
                "swizzle atoms need 1 KiB alignment");
  static_assert(SMEM <= 232448, "shared memory per CTA");
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
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void st_shared_zero16(uint32_t dst) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(dst), "r"(0u) : "memory");
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
// Four 8x8 bf16 matrices, transposed on the way out: register m of thread T holds row T/4, columns
// 2(T%4) and 2(T%4)+1 (low half first) of matrix m, and row r of matrix m is stored as column r, 16
// contiguous bytes at the address that thread 8m + r supplies.
__device__ __forceinline__ void stmatrix_x4_trans(uint32_t addr, uint32_t r0, uint32_t r1, uint32_t r2, uint32_t r3) {
  asm volatile("stmatrix.sync.aligned.m8n8.x4.trans.shared.b16 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(r0), "r"(r1),
               "r"(r2), "r"(r3)
               : "memory");
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// One MMA; the shared-memory descriptors are passed as their two 32-bit words (the high word is the
// same for every operand of this kernel, see desc_lo / kDescHi).
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo, uint32_t d_hi, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b64 da, db;\n\tsetp.ne.b32 p, %5, 0;\n\t"
      "mov.b64 da, {%1, %3};\n\tmov.b64 db, {%2, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %4, p;\n\t}" ::"r"(d_tmem),
      "r"(a_lo), "r"(b_lo), "r"(d_hi), "r"(idesc), "r"(accumulate)
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

// The 128-token x 32-column S tile of this warp's 32 TMEM lanes in the 16x256b shape (two loads of
// 16 lanes): thread T holds tokens 8z + T/4 (z = 0..3, relative to the warp's first lane) and columns
// 8k + 2(T%4) + e (k = 0..3, e = 0..1), in register sidx(z, k, e).
__device__ __forceinline__ constexpr int sidx(int z, int k, int e) { return (z >> 1) * 16 + k * 4 + (z & 1) * 2 + e; }
__device__ __forceinline__ void tmem_ld_s(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x4.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%32];\n\t"
      "tcgen05.ld.sync.aligned.16x256b.x4.b32 {%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, "
      "[%33];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr), "r"(taddr + (16u << 16))
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
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

// Shared-memory matrix descriptor, 128-byte swizzle (atoms of 8 rows x 128 B), as two 32-bit words.
// Low word: start address / 16 (bits 0-13) and the leading-dimension byte offset / 16 (bits 16-29).
// High word (descriptor bits 32-63): stride byte offset / 16 = 1024 / 16 (8-row groups 1 KiB apart),
// the tcgen05 descriptor version (bit 46) and the 128-byte swizzle mode (2 in bits 61-63).
constexpr uint32_t kDescHi = (1024u >> 4) | (1u << (46 - 32)) | (2u << (61 - 32));
__device__ __forceinline__ uint32_t desc_lo(uint32_t saddr, uint32_t lbo_bytes) {
  return ((saddr >> 4) & 0x3FFFu) | (((lbo_bytes >> 4) & 0x3FFFu) << 16);
}
// The start-address field advanced by `bytes` (16-byte multiple; shared addresses stay below 256 KiB,
// so the field never carries into the next one).
__device__ __forceinline__ constexpr uint32_t desc_adv(uint32_t bytes) { return bytes >> 4; }

// Byte offset of 16-byte piece `chunk` (0..15 along the 128 dimensions) of row
// `row` in a K-major, 128-byte-swizzled [rows][128] bf16 tile: two atoms
// columns of 64 dimensions, `half_bytes` apart.
__device__ __forceinline__ uint32_t swz_offset(int row, int chunk, uint32_t half_bytes) {
  return static_cast<uint32_t>(chunk >> 3) * half_bytes + static_cast<uint32_t>(row) * 128u +
         (static_cast<uint32_t>((chunk & 7) ^ (row & 7)) << 4);
}

struct Seg {
  int part, g, rb, slot;
  int64_t tile0;   // first tile of the segment within its part
  int64_t n_tiles;
};

// Even split of the T tiles of a launch over G CTAs in 32-bit arithmetic (the host keeps T below
// 2^31): CTA k holds tiles [begin(k), begin(k + 1)) with begin(k) = floor(k T / G) = k q + floor(k r / G)
// for T = q G + r -- the same split as cta_tile_begin.
struct Split {
  uint32_t T, G, q, r;
  __device__ Split(uint32_t t, uint32_t g) : T(t), G(g), q(t / g), r(t % g) {}
  __device__ uint32_t begin(uint32_t k) const { return k * q + (k * r) / G; }
  // the CTA holding tile x: the largest k with begin(k) <= x (a float estimate, then exact steps)
  __device__ uint32_t cta_of(uint32_t x) const {
    uint32_t k = static_cast<uint32_t>(static_cast<float>(x) * (static_cast<float>(G) / static_cast<float>(T)));
    if (k >= G) k = G - 1;
    while (k + 1 < G && begin(k + 1) <= x) ++k;
    while (k > 0 && begin(k) > x) --k;
    return k;
  }
};

// The segment of this CTA that starts at tile x of its group's sequence (the tiles of every part
// for the group's head and row block): it runs to the end of the part or to the end of the CTA's range.
__device__ __forceinline__ Seg seg_at(const ChunkParams& P, const Split& sp, int grp, int64_t x64, int64_t x_end,
                                      int& hint) {
  const uint32_t x = static_cast<uint32_t>(x64);
  int i = hint;
  while (i + 1 < P.n_parts && static_cast<uint32_t>(P.parts[i + 1].tile_base) <= x) ++i;
  hint = i;
  const uint32_t nt = (static_cast<uint32_t>(P.parts[i].n_tok) + TOK - 1) / TOK;
  const uint32_t first = static_cast<uint32_t>(P.parts[i].tile_base);
  Seg s;
  s.part = i;
  s.g = grp / P.n_rowblk;
  s.rb = grp - s.g * P.n_rowblk;
  s.tile0 = x - first;
  s.n_tiles = min(x_end, static_cast<int64_t>(first) + nt) - x64;
  s.slot = static_cast<int>(static_cast<uint32_t>(blockIdx.x - grp * P.ctas_per_group) - sp.cta_of(first));
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
        atomicOr(err, kErrWait);
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
          atomicOr(err, kErrWait);
          return false;
        }
      }
    }
  }
};

// NK: 8-column blocks of S computed per warpgroup (query rows 0 .. 8*NK-1 of its 32); every pass has
// at most 8*NK valid rows per warpgroup.  DH: the head dimension, 64 or 128.
template <int MODE, int NK, int DH>
__global__ void __launch_bounds__(TcCfg<MODE>::THREADS, 1) chunk_attn_tc(const __grid_constant__ ChunkParams P) {
  static_assert(DH == 64 || DH == TILE_D, "head dimension");
  constexpr bool PAIR = MODE == kHeadPair;
  static_assert(!PAIR || DH == 64, "head pairs need head dimension 64");
  constexpr int TD = PAIR ? TILE_D : DH;  // dimensions of a tile row that are loaded and multiplied
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
  const uint32_t KFULL = bar0, KEMPTY = KFULL + 8u * C::KST, VFULL = KEMPTY + 8u * C::KST,
                 VEMPTY = VFULL + 8u * C::VST;
  const uint32_t SFULL = VEMPTY + 8u * C::VST, SEMPTY = SFULL + 16u, PFULL = SEMPTY + 16u, OFULL = PFULL + 16u,
                 OEMPTY = OFULL + 16u, QFULL = OEMPTY + 16u,
                 DRAIN = QFULL + 8u;
  volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(gbase + C::OFF_MISC);
  float* red = reinterpret_cast<float*>(gbase + C::OFF_RED);
  float* mnew = reinterpret_cast<float*>(gbase + C::OFF_MNEW);
  float* alpha = reinterpret_cast<float*>(gbase + C::OFF_ALPHA);
  float* fin = reinterpret_cast<float*>(gbase + C::OFF_FIN);
  const RowState* hdr = reinterpret_cast<const RowState*>(gbase + C::OFF_HDR);

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::KST; ++s) {
      mbar_init(KFULL + 8u * s, 32);
      mbar_init(KEMPTY + 8u * s, 1);
    }
    for (int s = 0; s < C::VST; ++s) {
      mbar_init(VFULL + 8u * s, 32);
      mbar_init(VEMPTY + 8u * s, 1);
    }
    for (int b = 0; b < 2; ++b) {  // tile parity
      mbar_init(SFULL + 8u * b, 1);
      mbar_init(SEMPTY + 8u * b, 128 * NWG);
      mbar_init(PFULL + 8u * b, 128 * NWG);
      mbar_init(OFULL + 8u * b, 1);
      mbar_init(OEMPTY + 8u * b, 128 * NWG);
    }
    mbar_init(QFULL, 128 * NWG);
    mbar_init(DRAIN, 1);
    misc[1] = 0u;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    fence_proxy_async();
  }
  if constexpr (TD < TILE_D) {
    // the upper 64 dimensions of every V slot stay zero for the whole launch (the producers write only
    // the lower half), so the PV product's rows 64..127 are zero
    for (uint32_t o = threadIdx.x * 16u; o < static_cast<uint32_t>(C::VST * HALF_BYTES); o += C::THREADS * 16u)
      st_shared_zero16(base + C::OFF_V + (o / HALF_BYTES) * TILE_BYTES + HALF_BYTES + o % HALF_BYTES);
    fence_proxy_async();  // generic-proxy stores, later read by the tensor cores
  }
  if (warp == 0) tmem_alloc(base + C::OFF_MISC, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  // everything above touched only shared memory and TMEM; global memory only after the kernel
  // before this one in the stream has completed
  grid_dependency_wait();
  Waiter W{misc + 1, P.err};

  const int64_t T = P.total_tiles;
  // this CTA's group (KV head, row block) and its share of the group's tiles; CTA j of every group
  // covers the same token ranges, so the heads of a request are read in step
  const int grp = static_cast<int>(blockIdx.x) / P.ctas_per_group;
  const uint32_t jg = blockIdx.x - static_cast<uint32_t>(grp * P.ctas_per_group);
  const Split split(static_cast<uint32_t>(T), static_cast<uint32_t>(P.ctas_per_group));
  const int64_t x_begin = split.begin(jg);
  const int64_t x_end = split.begin(jg + 1);
  const int64_t kv_stride = static_cast<int64_t>(P.n_kv_heads) * DH;

  if (warp == 4 * NWG || warp == 4 * NWG + 1) {
    // ---------------- producers: warp 4*NWG fills the K ring, warp 4*NWG+1 the V ring
    const bool is_v = warp == 4 * NWG + 1;
    const int nst = is_v ? C::VST : C::KST;
    const uint32_t ring = base + (is_v ? C::OFF_V : C::OFF_K);
    const uint32_t full = is_v ? VFULL : KFULL, empty = is_v ? VEMPTY : KEMPTY;
    int hint = 0;
    int64_t i = 0;
    bool ok = true;
    for (int64_t x = x_begin; x < x_end && ok;) {
      const Seg sg = seg_at(P, split, grp, x, x_end, hint);
      const PartDesc& pd = P.parts[sg.part];
      const int64_t n_tok = pd.n_tok;
      // a group's head (or, for head pairs, pair p: heads 2p and 2p + 1, dimensions 128p .. 128p + 127)
      const __nv_bfloat16* const kv_base = is_v ? pd.v : pd.k;
      const __nv_bfloat16* src = kv_base + static_cast<int64_t>(sg.g) * TD;
      for (int64_t t = 0; t < sg.n_tiles; ++t, ++i) {
        const int slot = static_cast<int>(i % nst);
        const uint32_t use = static_cast<uint32_t>(i / nst);
        if (i >= nst && !W.wait(empty + 8u * slot, (use - 1u) & 1u)) {
          ok = false;
          break;
        }
        const int64_t tok0 = (sg.tile0 + t) * TOK;
        const uint32_t dst = ring + static_cast<uint32_t>(slot) * TILE_BYTES;
        // a token row of one head is PC 16-byte pieces; lane copies piece c = lane % PC of rows
        // r0 + RPI*j (j < TOK/RPI); rows past n_tok read nothing
        constexpr int PC = TD / 8, RPI = 32 / PC;
        const int c = lane % PC, r0 = lane / PC;
        int64_t valid_rows = (n_tok - tok0 < TOK) ? (n_tok - tok0) : static_cast<int64_t>(TOK);
        // (checked build) the tile's rows of this head lie in the part; else nothing is read
        if (!in_bounds(src + tok0 * kv_stride, (valid_rows - 1) * kv_stride + TD, kv_base, n_tok * kv_stride, P.err,
                       kSiteTcKV))
          valid_rows = 0;
        const __nv_bfloat16* ps = src + (tok0 + r0) * kv_stride + c * 8;
        const int64_t step = RPI * kv_stride;
        const uint32_t so0 = static_cast<uint32_t>(c >> 3) * HALF_BYTES + static_cast<uint32_t>(r0) * 128u;
        if (valid_rows == TOK) {
#pragma unroll 16
          for (int j = 0; j < TOK / RPI; ++j) {
            const int row = r0 + RPI * j;
            cp_async16(dst + so0 + static_cast<uint32_t>(j) * (RPI * 128u) +
                           (static_cast<uint32_t>((c & 7) ^ (row & 7)) << 4),
                       ps, 16);
            ps += step;
          }
        } else {
#pragma unroll 8
          for (int j = 0; j < TOK / RPI; ++j) {
            const int row = r0 + RPI * j;
            const bool in = row < valid_rows;
            cp_async16(dst + so0 + static_cast<uint32_t>(j) * (RPI * 128u) +
                           (static_cast<uint32_t>((c & 7) ^ (row & 7)) << 4),
                       in ? ps : src, in ? 16 : 0);
            ps += step;
          }
        }
        cp_async_arrive_noinc(full + 8u * slot);
      }
      x += sg.n_tiles;
    }
    cp_async_wait_all();
  } else if (warp == 4 * NWG + 2) {
    // ---------------- MMA issuer (one thread)
    if (lane == 0) {
      constexpr int ROWS = C::ROWS;
      constexpr uint32_t idesc_s = make_idesc(128, ROWS, false, false);
      constexpr uint32_t idesc_o = make_idesc(128, ROWS, true, false);
      const uint32_t qa = desc_lo(base + C::OFF_Q, 16);
      // S^T of tile j: K tile (A, K-major) x the pass's Q rows (B, K-major)
      auto issue_s = [&](int64_t j) {
        const int slot = static_cast<int>(j % C::KST);
        const uint32_t kaddr = base + C::OFF_K + static_cast<uint32_t>(slot) * TILE_BYTES;
        fence_proxy_async();  // cp.async writes (generic proxy) before tensor-core reads (async proxy)
        tc_fence_after();
        const uint32_t d = tmem + C::S_COL + static_cast<uint32_t>(j & 1) * ROWS;
        const uint32_t ka = desc_lo(kaddr, 16);
#pragma unroll
        for (int kk = 0; kk < TD / 16; ++kk)
          mma_bf16(d, ka + desc_adv((kk >> 2) * HALF_BYTES + (kk & 3) * 32),
                   qa + desc_adv((kk >> 2) * (ROWS * 128) + (kk & 3) * 32), kDescHi, idesc_s, kk > 0 ? 1u : 0u);
        mma_commit(SFULL + 8u * static_cast<uint32_t>(j & 1));
        mma_commit(KEMPTY + 8u * static_cast<uint32_t>(slot));  // the K slot is free when this fires
      };
      // O^T of tile j: V tile (A, dimension-major) x P^T (B, K-major)
      auto issue_pv = [&](int64_t j) {
        const int slot = static_cast<int>(j % C::VST);
        const uint32_t vaddr = base + C::OFF_V + static_cast<uint32_t>(slot) * TILE_BYTES;
        const uint32_t paddr = base + C::OFF_P + static_cast<uint32_t>(j & 1) * C::P_BYTES;
        fence_proxy_async();  // P^T was written with ordinary stores
        tc_fence_after();
        const uint32_t d = tmem + C::O_COL + static_cast<uint32_t>(j & 1) * ROWS;
        // A = V^T: 64-dimension halves 16 KiB apart (LBO), 8-token groups 1 KiB apart (SBO)
        const uint32_t va = desc_lo(vaddr, HALF_BYTES), pa = desc_lo(paddr, 16);
#pragma unroll
        for (int kk = 0; kk < TOK / 16; ++kk)
          mma_bf16(d, va + desc_adv(kk * 2048), pa + desc_adv((kk >> 2) * (ROWS * 128) + (kk & 3) * 32), kDescHi,
                   idesc_o, kk > 0 ? 1u : 0u);
        mma_commit(OFULL + 8u * static_cast<uint32_t>(j & 1));
        mma_commit(VEMPTY + 8u * static_cast<uint32_t>(slot));  // the V slot (and P^T buffer) is free when this fires
      };
      // Issue whichever product is ready, so a tile's PV never waits behind the next tile's data.
      // S(j) needs tile j's data, its segment's Q (first tile of a segment) and S buffer j&1 read by
      // the softmax (tile j-2); PV(j) needs S(j) issued, P^T(j) written and O buffer j&1 read (tile j-2).
      const int64_t n_local = x_end - x_begin;
      int64_t sn = 0, pn = 0;   // next tile (CTA-local) for S and for PV
      int64_t seg_end = 0;      // end of the segment S is in; sn == seg_end: S waits for the next Q
      uint32_t seg_idx = 0;
      int hint = 0;
      uint32_t spins = 0;
      uint64_t t_idle = 0;
      while (pn < n_local) {
        bool progress = false;
        if (sn < n_local) {
          if (sn == seg_end && mbar_test(QFULL, seg_idx & 1u)) {
            seg_end = sn + seg_at(P, split, grp, x_begin + sn, x_end, hint).n_tiles;
            ++seg_idx;
            tc_fence_after();
          }
          if (sn < seg_end && mbar_test(KFULL + 8u * static_cast<uint32_t>(sn % C::KST),
                                        static_cast<uint32_t>(sn / C::KST) & 1u) &&
              (sn < 2 || mbar_test(SEMPTY + 8u * static_cast<uint32_t>(sn & 1),
                                   (static_cast<uint32_t>(sn >> 1) & 1u) ^ 1u))) {
            issue_s(sn++);
            progress = true;
          }
        }
        if (pn < sn && mbar_test(PFULL + 8u * static_cast<uint32_t>(pn & 1), static_cast<uint32_t>(pn >> 1) & 1u) &&
            mbar_test(VFULL + 8u * static_cast<uint32_t>(pn % C::VST), static_cast<uint32_t>(pn / C::VST) & 1u) &&
            (pn < 2 ||
             mbar_test(OEMPTY + 8u * static_cast<uint32_t>(pn & 1), (static_cast<uint32_t>(pn >> 1) & 1u) ^ 1u))) {
          issue_pv(pn++);
          progress = true;
        }
        if (progress) {
          spins = 0;
        } else if ((++spins & 255u) == 0) {  // bounded: give up after kWaitLimitNs without progress
          if (*W.abort) break;
          const uint64_t now = global_ns();
          if (spins == 256u) {
            t_idle = now;
          } else if (now - t_idle > kWaitLimitNs) {
            *W.abort = 1u;
            atomicOr(W.err, kErrWait);
            break;
          }
        }
      }
      // drain: every MMA issued by this thread has completed before TMEM is freed
      mma_commit(DRAIN);
      W.drain(DRAIN, 0u);
    }
    __syncwarp();
  } else {
    // ---------------- softmax and accumulation: warpgroup wg = warp / 4.  For S tiles a thread holds
    // 4 tokens x 8 columns (16x256b TMEM shape, see tmem_ld_s); for O tiles it holds output
    // dimension tid, all 32 columns (32x32b shape).
    const int wg = warp >> 2;
    const int q4 = warp & 3;  // warp within the warpgroup: TMEM lanes / tile tokens 32*q4 .. 32*q4+31
    const int tid = threadIdx.x & 127;
    const uint32_t bar_wg = 1u + static_cast<uint32_t>(wg);
    const uint32_t lane_base = static_cast<uint32_t>(q4 * 32) << 16;
    constexpr int NC = 8 * NK;  // columns (query rows) computed: the active 8-column blocks
    float acc[NCOL];   // O^T accumulator: output dimension tid, query row c
    float s[32];       // S fragment, then the O^T tile values
    float negm[2 * NK];  // -reference maximum of the thread's columns 8k + 2(lane%4) + e, index 2k + e
    float thr[2 * NK];   // raw-score threshold of those columns: (reference + kTau) / scale
    float lsum[2 * NK];  // the thread's share of those columns' denominators (relative to the reference)
    const float inv_scale = 1.0f / P.q_scale;
    uint32_t rescaled = 0u;  // bit k: the tile with alpha buffer k re-based the row maxima
    float* red_w = red + wg * 4 * NCOL;
    float* mref = mnew + wg * NCOL;  // running reference maximum per row, shared by the warpgroup
    float* alpha_w = alpha + wg * 2 * NCOL;
    float* fin_w = fin + wg * 2 * NCOL;
    const RowState* hdr_w = hdr + wg * NCOL;  // the slot's previous headers of this warpgroup's rows
    const uint32_t hdr_s = base + C::OFF_HDR + static_cast<uint32_t>(wg * NCOL) * 16u;
    // shared address of row lane%8 of P^T matrix lane/8 (token block 4*q4 + lane/8) for column block 0
    // (the pass's P^T has C::ROWS rows; this warpgroup's start at row wg * NCOL)
    const int tb = 4 * q4 + (lane >> 3), pr = lane & 7;
    const uint32_t p_thread = static_cast<uint32_t>(tb >> 3) * (C::ROWS * 128) +
                              static_cast<uint32_t>(wg * NCOL + pr) * 128u + (static_cast<uint32_t>((tb & 7) ^ pr) << 4);
    const uint32_t col_wg = static_cast<uint32_t>(wg * NCOL);  // this warpgroup's columns in S and O
    int hint = 0;
    int64_t i = 0;
    bool ok = true;
    int nr = NCOL;
    auto abuf = [](int64_t j) { return static_cast<int>(j & 1); };

    auto accumulate = [&](int64_t j) -> bool {
      const uint32_t par = static_cast<uint32_t>(j & 1);
      if (!bar_all(bar_wg, 128, W.wait(OFULL + 8u * par, static_cast<uint32_t>(j >> 1) & 1u))) return false;
      tc_fence_after();
      tmem_ld32<0>(tmem + lane_base + C::O_COL + par * C::ROWS + col_wg, s);
      tc_fence_before();
      mbar_arrive(OEMPTY + 8u * par);
      if ((rescaled >> abuf(j)) & 1u) {
        const float4* al4 = reinterpret_cast<const float4*>(alpha_w + abuf(j) * NCOL);
#pragma unroll
        for (int c4 = 0; c4 < NC / 4; ++c4) {
          const float4 a = al4[c4];
          acc[4 * c4 + 0] = fmaf(acc[4 * c4 + 0], a.x, s[4 * c4 + 0]);
          acc[4 * c4 + 1] = fmaf(acc[4 * c4 + 1], a.y, s[4 * c4 + 1]);
          acc[4 * c4 + 2] = fmaf(acc[4 * c4 + 2], a.z, s[4 * c4 + 2]);
          acc[4 * c4 + 3] = fmaf(acc[4 * c4 + 3], a.w, s[4 * c4 + 3]);
        }
      } else {
#pragma unroll
        for (int c = 0; c < NC; ++c) acc[c] += s[c];
      }
      return true;
    };

    // This warpgroup's 32 Q rows of a pass into shared memory (K-major swizzled [ROWS][128], padding
    // rows zero; with d = 64 and one head per group the upper half is never read) with cp.async; QFULL
    // completes when every softmax thread's copies have landed.  Head pairs: warpgroup wg's rows are head
    // 2p + wg's, written into dimension half wg, and the other half is zero-filled.
    int hint_q = 0;
    auto load_q = [&](int64_t xq) {
      const Seg sq = seg_at(P, split, grp, xq, x_end, hint_q);
      if constexpr (PAIR) {
        int nrows = min(NCOL, P.group * P.n_query);
        const int64_t qrow0 = (static_cast<int64_t>(P.parts[sq.part].req) * P.n_q_heads +
                               static_cast<int64_t>(2 * sq.g + wg) * P.group) * P.n_query;
        if (!in_bounds(P.q + qrow0 * DH, static_cast<int64_t>(nrows) * DH, P.q, P.q_rows * DH, P.err, kSiteTcQ)) nrows = 0;
#pragma unroll
        for (int idx = tid; idx < NCOL * (TILE_D / 8); idx += 128) {
          const int r = idx / (TILE_D / 8), ch = idx % (TILE_D / 8);
          const bool in = r < nrows && (ch >> 3) == wg;
          cp_async16(base + C::OFF_Q + swz_offset(wg * NCOL + r, ch, C::ROWS * 128),
                     in ? P.q + (qrow0 + r) * DH + (ch & 7) * 8 : P.q, in ? 16 : 0);
        }
      } else {
        const int rblk = sq.rb * C::ROWS;
        int nrows = min(C::ROWS, P.group * P.n_query - rblk);
        const int64_t qrow0 = (static_cast<int64_t>(P.parts[sq.part].req) * P.n_q_heads +
                               static_cast<int64_t>(sq.g) * P.group) * P.n_query + rblk;
        if (!in_bounds(P.q + qrow0 * DH, static_cast<int64_t>(nrows) * DH, P.q, P.q_rows * DH, P.err, kSiteTcQ)) nrows = 0;
#pragma unroll
        for (int idx = tid; idx < NCOL * (DH / 8); idx += 128) {
          const int c = wg * NCOL + idx / (DH / 8), ch = idx % (DH / 8);
          const bool in = c < nrows;
          cp_async16(base + C::OFF_Q + swz_offset(c, ch, C::ROWS * 128), in ? P.q + (qrow0 + c) * DH + ch * 8 : P.q,
                     in ? 16 : 0);
        }
      }
      cp_async_arrive_noinc(QFULL);
    };
    bool q_loaded = false;  // the current segment's Q was fetched during the previous segment

    for (int64_t x = x_begin; x < x_end;) {
      // all softmax threads meet here, so a wait that gave up anywhere stops every warpgroup together
      if (!bar_all(3u, 128u * NWG, ok)) break;
      const Seg sg = seg_at(P, split, grp, x, x_end, hint);
      const PartDesc& pd = P.parts[sg.part];
      const int b = pd.req;
      const int R = P.group * P.n_query;
      const int rblk = sg.rb * C::ROWS;                          // first row of this pass
      // this warpgroup's first row (of its head's rows; head pairs: each warpgroup has its own head)
      const int r0 = PAIR ? 0 : rblk + ((MODE == kRowSplit) ? wg * NCOL : 0);
      nr = max(0, min(NCOL, R - r0));
      const int head = PAIR ? 2 * sg.g + wg : sg.g;
      const int64_t qrow0 =
          (static_cast<int64_t>(b) * P.n_q_heads + static_cast<int64_t>(head) * P.group) * P.n_query;

      // this segment's state slot rows; their headers (written by earlier launches of the round, or stale)
      // are fetched now and read back at the segment's end (~1 us off the launch's tail)
      const int slot = P.slot_base + sg.slot;
      const int64_t srow0 = static_cast<int64_t>(slot) * P.slot_stride + qrow0 + r0;
      // (checked build) this warpgroup's state rows lie in the workspace; else they are neither read nor written
      const bool st_ok = in_bounds(P.ws_h + srow0, nr, P.ws_h, kHistSlots * P.slot_stride, P.err, kSiteTcState);
      if (tid < nr && st_ok) cp_async16(hdr_s + static_cast<uint32_t>(tid) * 16u, P.ws_h + srow0 + tid, 16);
      if (!q_loaded) load_q(x);
      q_loaded = false;
      if (q4 == 0) mref[lane] = -INFINITY;

#pragma unroll
      for (int c = 0; c < NCOL; ++c) acc[c] = 0.f;
#pragma unroll
      for (int j = 0; j < 2 * NK; ++j) {
        negm[j] = 0.f;
        thr[j] = -INFINITY;  // the first tile always re-bases
        lsum[j] = 0.f;
      }
      int64_t prev = -1;  // this warpgroup's previous tile in the segment
      const int64_t n_tok = pd.n_tok;

      for (int64_t t = 0; t < sg.n_tiles; ++t, ++i) {
        const uint32_t par = static_cast<uint32_t>(i & 1);
        if (!bar_all(bar_wg, 128, W.wait(SFULL + 8u * par, static_cast<uint32_t>(i >> 1) & 1u))) {
          ok = false;
          break;
        }
        tc_fence_after();
        tmem_ld_s(tmem + lane_base + C::S_COL + par * C::ROWS + col_wg, s);
        tc_fence_before();
        mbar_arrive(SEMPTY + 8u * par);

        // tokens past the part's end (last tile only) score -inf: they never vote and p = 0
        const int64_t tile_tok0 = (sg.tile0 + t) * TOK;
        if (tile_tok0 + TOK > n_tok) {
          const int64_t tok = tile_tok0 + 32 * q4 + (lane >> 2);
#pragma unroll
          for (int z = 0; z < 4; ++z) {
            const bool valid = tok + 8 * z < n_tok;
#pragma unroll
            for (int k = 0; k < NK; ++k) {
              s[sidx(z, k, 0)] = valid ? s[sidx(z, k, 0)] : -INFINITY;
              s[sidx(z, k, 1)] = valid ? s[sidx(z, k, 1)] : -INFINITY;
            }
          }
        }
        // does any score exceed its row's reference by more than kTau?
        bool up = false;
#pragma unroll
        for (int k = 0; k < NK; ++k)
#pragma unroll
          for (int z = 0; z < 4; ++z) {
            up |= s[sidx(z, k, 0)] > thr[2 * k];
            up |= s[sidx(z, k, 1)] > thr[2 * k + 1];
          }
        up = bar_any(bar_wg, 128, up);
        const int ab = abuf(i);
        rescaled = (rescaled & ~(1u << ab)) | (static_cast<uint32_t>(up) << ab);
        if (up) {
          // exact tile maximum per row: the thread's 4 tokens, the 8 lanes sharing the columns, the 4 warps
          float mx[2 * NK];
#pragma unroll
          for (int k = 0; k < NK; ++k)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              float v = fmaxf(fmaxf(s[sidx(0, k, e)], s[sidx(1, k, e)]), fmaxf(s[sidx(2, k, e)], s[sidx(3, k, e)]));
              v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
              v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
              v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
              mx[2 * k + e] = v;
            }
          if (lane < 4) {
#pragma unroll
            for (int k = 0; k < NK; ++k) {
              red_w[q4 * NCOL + 8 * k + 2 * lane] = mx[2 * k];
              red_w[q4 * NCOL + 8 * k + 2 * lane + 1] = mx[2 * k + 1];
            }
          }
          bar_sync(bar_wg, 128);
          if (q4 == 0 && lane < NC) {
            const int c = lane;
            const float tm =
                fmaxf(fmaxf(red_w[c], red_w[NCOL + c]), fmaxf(red_w[2 * NCOL + c], red_w[3 * NCOL + c])) * P.q_scale;
            const float mo = mref[c];
            const float mn = fmaxf(mo, tm);
            alpha_w[ab * NCOL + c] = (mo == -INFINITY) ? 0.f : exp2_approx(mo - mn);
            mref[c] = mn;
          }
          bar_sync(bar_wg, 128);
#pragma unroll
          for (int k = 0; k < NK; ++k)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int c = 8 * k + 2 * (lane & 3) + e;
              const float m = mref[c];
              negm[2 * k + e] = -m;
              thr[2 * k + e] = (m + kTau) * inv_scale;
              lsum[2 * k + e] *= alpha_w[ab * NCOL + c];
            }
        }

        // P^T = 2^(s*scale - m) in bf16, into the K-major swizzled B operand of the PV product (buffer
        // i&1, last read by PV(i-2), which completed before accumulate(i-2) ran): one 8-column block per
        // stmatrix, its four 8x8 matrices being the thread's four 8-token blocks
        const uint32_t pbase = base + C::OFF_P + static_cast<uint32_t>(i & 1) * C::P_BYTES + p_thread;
#pragma unroll
        for (int k = 0; k < NK; ++k) {
          uint32_t pk[4];
#pragma unroll
          for (int z = 0; z < 4; ++z) {
            const float p0 = exp2_approx(fmaf(s[sidx(z, k, 0)], P.q_scale, negm[2 * k]));
            const float p1 = exp2_approx(fmaf(s[sidx(z, k, 1)], P.q_scale, negm[2 * k + 1]));
            lsum[2 * k] += p0;
            lsum[2 * k + 1] += p1;
            pk[z] = pack_bf16x2(p0, p1);
          }
          stmatrix_x4_trans(pbase + static_cast<uint32_t>(k) * 1024u, pk[0], pk[1], pk[2], pk[3]);
        }
        fence_proxy_async();
        mbar_arrive(PFULL + 8u * par);
        // the segment's last S product has completed, so nothing reads Q any more: fetch the next
        // segment's Q now, and the MMAs can start on it while this segment's state is written
        if (t + 1 == sg.n_tiles && x + sg.n_tiles < x_end) {
          load_q(x + sg.n_tiles);
          q_loaded = true;
        }

        // the previous tile's O one step behind, so the MMAs of tile i overlap the accumulation
        if (prev >= 0 && !accumulate(prev)) {
          ok = false;
          break;
        }
        prev = i;
      }
      if (ok && prev >= 0) ok = accumulate(prev);
      if (ok && prev >= 0 && st_ok) {
        // this warpgroup's segment state (m = mref, l = sum over threads, a = acc), merged into the
        // slot's state when that is from this round (an earlier launch of the round)
#pragma unroll
        for (int j = 0; j < 2 * NK; ++j) {
          float v = lsum[j];
          v += __shfl_xor_sync(0xffffffffu, v, 4);
          v += __shfl_xor_sync(0xffffffffu, v, 8);
          v += __shfl_xor_sync(0xffffffffu, v, 16);
          lsum[j] = v;
        }
        if (lane < 4) {
#pragma unroll
          for (int k = 0; k < NK; ++k) {
            red_w[q4 * NCOL + 8 * k + 2 * lane] = lsum[2 * k];
            red_w[q4 * NCOL + 8 * k + 2 * lane + 1] = lsum[2 * k + 1];
          }
        }
        cp_async_wait_all();
        bar_sync(bar_wg, 128);
        if (q4 == 0 && lane < NC) {
          const int c = lane;
          fin_w[c] = mref[c];
          fin_w[NCOL + c] = red_w[c] + red_w[NCOL + c] + red_w[2 * NCOL + c] + red_w[3 * NCOL + c];
        }
        bar_sync(bar_wg, 128);
        // per 8-row block: the earlier accumulators first (independent loads), then the merged values
        // (threads past the head dimension hold the zero rows of O^T; with head pairs, thread tid holds
        // dimension tid - 64 wg of its warpgroup's head, and the other half holds the other head's values)
        const int dim = PAIR ? tid - 64 * wg : tid;
        const bool dim_ok = dim >= 0 && dim < DH;
        float* ap = P.ws_a + srow0 * DH + (dim_ok ? dim : 0);
#pragma unroll
        for (int k = 0; k < NK && dim_ok; ++k) {
          float olda[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int c = 8 * k + e;
            olda[e] = (c < nr && hdr_w[c].epoch == P.epoch) ? ap[c * DH] : 0.f;
          }
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int c = 8 * k + e;
            if (c < nr) {
              const float m = fin_w[c], mo = hdr_w[c].m;
              float a = acc[c];
              if (hdr_w[c].epoch == P.epoch) {
                const float mn = fmaxf(mo, m);
                if (mn != -INFINITY) a = olda[e] * exp2_approx(mo - mn) + a * exp2_approx(m - mn);
              }
              ap[c * DH] = a;
            }
          }
        }
        if (tid < nr) {
          float m = fin_w[tid], l = fin_w[NCOL + tid];
          const RowState oldh = hdr_w[tid];
          if (oldh.epoch == P.epoch) {
            const float mn = fmaxf(oldh.m, m);
            if (mn != -INFINITY) {
              l = oldh.l * exp2_approx(oldh.m - mn) + l * exp2_approx(m - mn);
              m = mn;
            }
          }
          P.ws_h[srow0 + tid] = RowState{m, l, P.epoch, 0u};
        }
      }
      x += sg.n_tiles;
    }
    cp_async_wait_all();  // a Q prefetch still in flight (a wait gave up) lands before the CTA exits
  }

  // The next kernel in the stream may be scheduled once every CTA got here.  Not earlier: a launch can
  // run for milliseconds (streaming from host memory on a few SMs), and waiting dependents would hold
  // the other SMs' resources against work on other streams.
  allow_dependents();
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int MODE, int NK, int DH>
cudaError_t launch_tc(const ChunkParams& p, int n_ctas, cudaStream_t stream) {
  using C = TcCfg<MODE>;
  static bool configured = false;
  if (!configured) {
    cudaError_t e =
        cudaFuncSetAttribute(chunk_attn_tc<MODE, NK, DH>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  return launch_pdl(chunk_attn_tc<MODE, NK, DH>, dim3(n_ctas), dim3(C::THREADS), C::SMEM, stream, p);
}

template <int DH>
cudaError_t launch_tc_dh(const ChunkParams& p, int mode, int n_ctas, cudaStream_t stream) {
  const int R = p.group * p.n_query;
  if (mode == kSingle) {  // one pass of R <= 32 rows: compute ceil(R / 8) column blocks
    if (R < 1 || R > TcCfg<kSingle>::ROWS) return cudaErrorInvalidValue;
    switch ((R + 7) / 8) {
      case 1: return launch_tc<kSingle, 1, DH>(p, n_ctas, stream);
      case 2: return launch_tc<kSingle, 2, DH>(p, n_ctas, stream);
      case 3: return launch_tc<kSingle, 3, DH>(p, n_ctas, stream);
      default: return launch_tc<kSingle, 4, DH>(p, n_ctas, stream);
    }
  }
  if (mode == kRowSplit) return launch_tc<kRowSplit, 4, DH>(p, n_ctas, stream);
  if constexpr (DH == 64) {
    if (mode == kHeadPair) {  // each head's R <= 32 rows: ceil(R / 8) column blocks
      if (R < 1 || R > TcCfg<kHeadPair>::NCOL) return cudaErrorInvalidValue;
      switch ((R + 7) / 8) {
        case 1: return launch_tc<kHeadPair, 1, 64>(p, n_ctas, stream);
        case 2: return launch_tc<kHeadPair, 2, 64>(p, n_ctas, stream);
        case 3: return launch_tc<kHeadPair, 3, 64>(p, n_ctas, stream);
        default: return launch_tc<kHeadPair, 4, 64>(p, n_ctas, stream);
      }
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace

bool tc_supported(int head_dim, int rows) { return (head_dim == 64 || head_dim == 128) && rows >= 1; }
int tc_mode(int rows) { return rows <= TcCfg<kSingle>::ROWS ? kSingle : kRowSplit; }
int tc_mode_for(int head_dim, int n_kv_heads, int rows) {
  if (head_dim == 64 && n_kv_heads % 2 == 0 && rows <= TcCfg<kHeadPair>::NCOL) return kHeadPair;
  return tc_mode(rows);
}
int tc_rows_per_pass(int mode) {
  if (mode == kRowSplit) return TcCfg<kRowSplit>::ROWS;
  return TcCfg<kSingle>::ROWS;  // kSingle; kHeadPair: the rows of one head per warpgroup
}
int tc_slots_per_segment(int) { return 1; }
int tc_max_ctas(int num_sms) { return num_sms; }  // one CTA per SM (shared memory)

int64_t tc_plan(ChunkParams& p, int mode, int64_t cta_budget, int64_t* slots) {
  const int R = p.group * p.n_query;
  const int rpp = tc_rows_per_pass(mode);
  p.n_rowblk = (R + rpp - 1) / rpp;
  // one CTA group per (head, row block), or per pair of heads; each group's tiles (that head and row
  // block of every part, part after part) are split evenly over its CTAs, so CTA j of every group
  // covers the same tokens
  const int64_t groups = mode == kHeadPair ? static_cast<int64_t>(p.n_kv_heads / 2)
                                           : static_cast<int64_t>(p.n_kv_heads) * p.n_rowblk;
  int64_t T = 0;
  for (int i = 0; i < p.n_parts; ++i) {
    p.parts[i].tile_base = T;
    T += (static_cast<int64_t>(p.parts[i].n_tok) + TOK - 1) / TOK;
  }
  p.total_tiles = T;
  auto segments = [&](int64_t cpg) {  // the most CTA segments any part spreads over
    int64_t worst = 0;
    for (int i = 0; i < p.n_parts; ++i) {
      const int64_t first = p.parts[i].tile_base, nt = (static_cast<int64_t>(p.parts[i].n_tok) + TOK - 1) / TOK;
      worst = std::max(worst, cta_of_tile(first + nt - 1, cpg, T) - cta_of_tile(first, cpg, T) + 1);
    }
    return worst;
  };
  int64_t cpg = std::min<int64_t>(std::max<int64_t>(1, cta_budget / groups), T);
  const int sps = tc_slots_per_segment(mode);
  while (cpg > 1 && segments(cpg) * sps > kHistSlots) --cpg;
  *slots = segments(cpg) * sps;
  p.ctas_per_group = static_cast<int32_t>(cpg);
  return groups * cpg;
}

cudaError_t launch_chunk_attn_tc(const ChunkParams& p, int head_dim, int mode, int n_ctas, cudaStream_t stream) {
  if (n_ctas < 1) return cudaSuccess;
  if (p.total_tiles > INT32_MAX) return cudaErrorInvalidValue;  // the kernel splits tiles in 32-bit arithmetic
  if (head_dim == 128) return launch_tc_dh<128>(p, mode, n_ctas, stream);
  if (head_dim == 64) return launch_tc_dh<64>(p, mode, n_ctas, stream);
  return cudaErrorInvalidValue;
}

}  // namespace svx
