// Causal prefill over the position-free paged cache on the 5th-generation tensor cores.
//
// [NOTE] Tiling 感知的 Q/K 旋转分派: in prefill the query tile is much taller than a KV tile,
// so the KV side is rotated: every staged K tile gets one relative rotation R_Delta per
// document (3 extra flops per K scalar) before the QK^T GEMM.  [NOTE] 融合 Triton kernel:
// the K tile is split in its two half-dimensions, rotated, then multiplied.  [GIST]
// Prefilling: a single relative rotation by the offset, never un-rotate then re-rotate.
//
// GB300 design.  One CTA per (request, KV head, 256 query rows) = two 128-row Q tiles that share
// every K/V tile, so each staged (and rotated) K tile and each V tile feeds twice the MMA work.
// 512 threads, 1 CTA per SM, registers re-split per warpgroup with setmaxnreg:
//   warps 0-3 / 4-7  softmax of Q tile 0 / 1 (thread r owns TMEM lane r = row r of its tile):
//              prepare the tile's Q rows (rotation by the absolute position m, softmax scale
//              folded in, 128B-swizzled K-major operand), then per K tile: S row from TMEM, mask,
//              online softmax in base 2 (the running max moves, and O is rescaled in TMEM, only
//              when a row's max grows by more than 8), P written back to TMEM over S as bf16.
//   warps 8-11 K rotation: each staged K tile's page rows rotated by their page's Delta in
//              place in shared memory; a thread owns one chunk pair (8 frequencies) of 8 rows of
//              a page and keeps their cos/sin in registers, recomputed when the Delta changes.
//   warp 12    producer: unpacks the 64-bit block words of a tile's 8 pages (prefetched one tile
//              ahead) and issues TMA loads (box 64 columns x 16 rows of one page, 128-byte
//              swizzle) into a 3-stage K ring (K runs two tiles ahead of V) and a 2-stage V
//              ring; in the SPLIT_V instantiation warp 14 issues V with its own barrier chain
//              (one live Q tile, long key ranges).  A page with r < 16 rows that hold a key
//              visible to the CTA (a document's partial last page, or query-segment rows past
//              the CTA's last token) is loaded from row r - 16: its r key rows land in the
//              stage's last r rows and the 16 - r rows before them are out of the tensor's
//              bounds, which TMA fills with zeros.  Bytes past a key are never read, so stale
//              or never-written cache rows (any bit pattern, NaN included) cannot reach PV,
//              where a zero weight times NaN would still be NaN.
//   warp 13    TMEM owner and MMA issuer, in the order QK0(j) QK1(j) | PV0(j) QK0(j+1) PV1(j)
//              QK1(j+1) | ...: S_i = Q_i K^T (A and B from shared memory) into TMEM, then
//              O_i += P_i V with P_i read from TMEM (A operand in tensor memory) and V as an
//              MN-major shared-memory operand.  The tensor pipe runs a thread's MMAs in issue
//              order, so S_i of tile j+1 is only written after PV_i(j) has read P_i, and the
//              commit that signals S_i(j+1) also covers PV_i(j).
// TMEM columns: S0 [0,128), S1 [128,256), O0 [256,384), O1 [384,512); P_i = first 64 of S_i.
// With one live Q tile (short queries, decode), S0 and S1 double-buffer that tile's scores
// instead (tile j in S_{j%2}), so QK^T of tile j+1 runs while the softmax works on tile j.  In
// launches whose CTAs all have one live Q tile (the KH instantiation) warps 0-3 and 4-7 each
// take half of every tile's keys (keys 0-63 / 64-127, P over the start of each half's own S
// columns): two partial softmaxes accumulated into O_A [256,384) and O_B [384,512) by two PV
// MMAs of 64 keys, merged by their maxima and sums in the epilogue.  A softmax warp thus does
// half the work per tile, and each SM sub-partition has two of them.
// GQA: a tile's rows are (token, head) pairs of the KV head's query-head group, token-major.
// Decode mode serves wide head groups (MQA): the G heads of one new token fill the rows, the
// key range is split over several CTAs and their partials are merged by log-sum-exp.
// With ALiBi the tiles are visited newest first (the running max is fixed by the first tile),
// and the bias -slope (m - p) is split into slope t per key row t of a page (a packed FMA on
// the scores) and slope (pstart - m) per page (on the page's max and its exponent offset).
// Every wait is bounded (mbarrier polls against %globaltimer; an abort flag ends all roles).
// Warp 15 has no role, nor has warp 14 outside SPLIT_V (or warps 4-7 of a CTA with one live
// Q tile outside KH).
#include <cfloat>
#include <climits>

#include <cuda.h>  // CUtensorMap and the encoder's types (the function is looked up at run time)

#include "common.cuh"

namespace lazykv {

namespace tc {

constexpr int kM = 128;            // query rows per Q tile
constexpr int kQT = 2;             // Q tiles per CTA
constexpr int kN = 128;            // keys per K/V tile
constexpr int kPagesPerTile = kN / kPage;
constexpr int kKStages = 3;        // K ring depth: K runs two tiles ahead of V
constexpr int kVStages = 2;        // V ring depth
constexpr int kSlots = 6;          // per-tile metadata slots (tile j uses slot j % 6): with K two
                                   // tiles ahead, tile j + 4 is published while the softmax of
                                   // tile j may still read its slot (one live Q tile)
constexpr int kThreads = 512;
constexpr int kRotWarp0 = 8;
constexpr int kProdWarp = 12;
constexpr int kMmaWarp = 13;
constexpr int kVProdWarp = 14;  // V producer of the SPLIT_V instantiation
// Registers per thread after the re-split, per warpgroup role (softmax, rotation, producer +
// MMA), chosen by the spills ptxas reports: kernels that rotate K give the rotation warps 56
// (48 spills there); two Q tiles keep a 128-score row per softmax thread (184 or 192), while
// with key halves a softmax thread holds 64 scores and 176 leave the producer and MMA warps
// enough to spill nothing.  Every split adds up to 512 * 128 = 65536.
constexpr int kRegsLaunch = 128;
template <bool ROT, bool KH = false> struct Regs {
  static constexpr int softmax = KH ? 176 : (ROT ? 184 : 192);
  static constexpr int rot = ROT ? 56 : 48;
  static constexpr int issue = KH ? (ROT ? 104 : 112) : (ROT ? 88 : 80);
  static_assert(2 * 128 * softmax + 128 * rot + 128 * issue == kThreads * kRegsLaunch,
                "warpgroup register shares must add up to the launch allocation");
};
constexpr float kTau = 8.0f;

// barrier indices
enum : int {
  B_K_FULL = 0,    // [3] K tile landed (TMA bytes)
  B_K_READY = 3,   // [3] K tile rotated (128 arrivals)
  B_K_FREE = 6,    // [3] both QK^T done with the K stage (commit)
  B_V_FULL = 9,    // [2] V tile landed (TMA bytes)
  B_V_FREE = 11,   // [2] both PV done with the V stage (commit)
  B_S_FULL = 13,   // [2] per Q tile (one live tile: per S buffer): S written (commit)
  B_P_FULL = 15,   // [2] per Q tile (one live tile: per S buffer): P in TMEM, O rescaled (128)
  B_Q_READY = 17,  // both Q tiles prepared (256 arrivals)
  B_FINAL = 18,    // all MMAs finished (commit)
  B_PV_DONE = 19,  // one live Q tile only: PV of a tile finished (commit)
  NBAR = 20
};
// Every waiter consumes every phase of the barriers it waits on, in order: a parity wait
// (mbarrier.try_wait.parity) cannot tell the phase it asks for from the one two phases
// earlier, so waiting on a later phase while an earlier one is still open passes at once.

template <int D>
struct Layout {
  static constexpr int CB = D / 64;                        // 128-byte column blocks per row
  static constexpr int BLK = kM * 128;                     // one column block of a 128-row tile
  static constexpr int TILE = kN * D * 2;                  // one K or V tile
  static constexpr int QTILE = kM * D * 2;                 // one Q tile
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = Q_OFF + kQT * QTILE;        // K ring
  static constexpr int V_OFF = K_OFF + kKStages * TILE;    // V ring
  static constexpr int PSTART_OFF = V_OFF + kVStages * TILE;  // int [slot][8] key position of stage row 0
  static constexpr int PINFO_OFF = PSTART_OFF + kSlots * kPagesPerTile * 4;  // int2 [slot][8] {Delta, lo}:
                                                                            // stage rows [lo, 16) hold keys
  static constexpr int FLAG_OFF = PINFO_OFF + kSlots * kPagesPerTile * 8;  // int [slot][2] {fast, pad}
  static constexpr int PGID_OFF = FLAG_OFF + kSlots * 8;                // int [slot][8] page * Hkv + head
  static constexpr int TURNS_OFF = PGID_OFF + kSlots * kPagesPerTile * 4;  // u64 [D/2]
  static constexpr int BAR_OFF = TURNS_OFF + (D / 2) * 8;
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;                   // tmem slot, abort flag
  static constexpr int SMEM = MISC_OFF + 16 + 1024;                     // + alignment slack
};
static_assert(Layout<128>::SMEM <= 227 * 1024, "shared memory budget");

struct Args {
  const __nv_bfloat16* q;
  const int32_t* cu_q;
  const int32_t* q_start;
  const int32_t* doc_blocks;
  const uint64_t* meta;
  int B, max_blocks, Hq, Hkv, num_pages;
  __nv_bfloat16* out;
  float* lse;
  uint32_t* status;
  PosParams pos;
  // decode mode (seq_len != null): one query row per request at m = seq_len - 1, the key range
  // split over S CTAs whose unnormalised partials (O, base-2 max, sum) go to part_o / part_ml
  const int32_t* seq_len;
  int S;
  float* part_o;   // [B][Hq][S][D]
  float* part_ml;  // [B][Hq][S][2]
};

// ---------------------------------------------------------------- tcgen05 / TMA wrappers
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  // tcgen05 shared-memory matrix descriptor: start>>4, LBO>>4, SBO>>4, version 1,
  // base offset 0 (1024-byte aligned atoms), 128-byte swizzle.
  return uint64_t((addr & 0x3FFFFu) >> 4) | (uint64_t((lbo >> 4) & 0x3FFFu) << 16) |
         (uint64_t((sbo >> 4) & 0x3FFFu) << 32) | (uint64_t(1) << 46) | (uint64_t(2) << 61);
}

// instruction descriptor, kind::f16: fp32 accumulate, A and B both bf16 (ab_f16 = 0) or both
// f16 (ab_f16 = 1), K-major A, B K-major (b_mn = 0) or MN-major (b_mn = 1), shape M x N.
__host__ __device__ constexpr uint32_t idesc_mma(int M, int N, int b_mn, int ab_f16) {
  return (1u << 4) | (uint32_t(ab_f16 ? 0 : 1) << 7) | (uint32_t(ab_f16 ? 0 : 1) << 10) | (uint32_t(b_mn) << 16) |
         (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}

__device__ __forceinline__ uint32_t f2_to_h2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
        "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
        "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
      "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]),
      "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]),
      "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 3-D tiled load (column x, row y inside the page, page-head z).  y may be negative: the rows of
// the box before row 0 are outside the tensor and arrive as zeros; the transaction still
// counts the whole box.  x is always a multiple of 64 elements (128 bytes).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void named_sync(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }

// Bounded wait that also gives up when another role has aborted.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag, uint32_t* status) {
  if (mbar_test(bar, parity)) return true;
  WaitClock clk;
  uint32_t n = 0;
  while (true) {
    if (mbar_test(bar, parity)) return true;
    if ((++n & 63u) == 0) {
      if (*abort_flag) return false;
      if (clk.expired()) {
        *abort_flag = 1;
        set_status(status, LAZY_STATUS_TIMEOUT);
        return false;
      }
    }
  }
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr)
               : "memory");
  return v;
}

// byte offset of 16-byte chunk c of row r inside a 128-byte-swizzled block (1024-byte atoms)
__device__ __forceinline__ uint32_t swz(int r, int c) { return uint32_t(r * 128 + ((c ^ (r & 7)) << 4)); }

// O += P V with P (the A operand, M x K, 16-bit pairs packed per 32-bit column) in TMEM
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

// ---------------------------------------------------------------- the kernel
__device__ __forceinline__ float max3f(float a, float b, float c) {  // three-input maximum
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

__device__ __forceinline__ float ex2(float x) {  // 2^x on the MUFU (approx, flush-to-zero)
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// SPLIT_V: with one live Q tile, V is issued by warp 14 with its own barrier chain instead of
// being interleaved behind K by warp 12.  Chosen on the host for long one-Q-tile key ranges
// (decode mode, long-context prefill with short queries), where V copies queued behind K leave
// the ingest short; the two-Q-tile schedule keeps one producer.  A separate instantiation, so
// each schedule's code is generated on its own.
template <int D, int POS, bool SPLIT_V, bool KH>
__global__ void __launch_bounds__(kThreads, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv, const Args a) {
  using L = Layout<D>;
  constexpr bool kRotate = (POS == kRope || POS == kRopeX);
  // With rotation, the rotated Q and K are rounded once more before QK^T: write them as f16
  // (10 mantissa bits; stored bf16 keys convert exactly) so QK^T runs as an f16 x f16 MMA.
  // Without rotation K is the stored bf16 itself, so Q is rounded to bf16.  PV is bf16 x bf16.
  constexpr bool kQkF16 = kRotate;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;
  uint8_t* sm = smem_raw + (sb - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = int(blockIdx.x) % a.S, mp = int(blockIdx.x) / a.S, g = blockIdx.y, b = blockIdx.z;
  pdl_wait();
  const int G = a.Hq / a.Hkv;
  const int tpt = kM / G;  // tokens per Q tile
  const int qs = a.q_start[b];
  const bool dec = a.seq_len != nullptr;
  const int q0 = dec ? b : a.cu_q[b];                      // first query row of the request
  const int Lq = dec ? 1 : a.cu_q[b + 1] - q0;
  const int mbase = dec ? a.seq_len[b] - 1 : qs;           // absolute position of its token 0
  const int tok0 = mp * kQT * tpt;
  if (tok0 >= Lq) return;  // uniform for the CTA, before any barrier or TMEM use
  const int nq = (tok0 + tpt < Lq) ? 2 : 1;  // live Q tiles
  const int ntok = min(kQT * tpt, Lq - tok0);
  const int m_min = mbase + tok0, m_max = mbase + tok0 + ntok - 1;
  int nb = a.doc_blocks[b] + (m_max - qs) / kPage + 1;
  if (nb > a.max_blocks) {
    if (threadIdx.x == 0) set_status(a.status, LAZY_STATUS_BAD_ROW);
    nb = a.max_blocks;
  }
  const int ntiles_all = (nb + kPagesPerTile - 1) / kPagesPerTile;
  const int chunk = (ntiles_all + a.S - 1) / a.S;
  const int t0 = split * chunk;                            // first K/V tile of this CTA
  const int ntiles = min(ntiles_all, t0 + chunk) - t0;
  if (ntiles <= 0) {  // an empty split contributes a neutral partial (uniform for the CTA)
    for (int i = threadIdx.x; i < ntok * G; i += blockDim.x) {
      const size_t pi = ((size_t)(q0 + tok0 + i / G) * a.Hq + g * G + i % G) * a.S + split;
      a.part_ml[pi * 2] = -INFINITY;
      a.part_ml[pi * 2 + 1] = 0.f;
      for (int c = 0; c < D; ++c) a.part_o[pi * D + c] = 0.f;
    }
    return;
  }

  const uint32_t sQ0 = sb + L::Q_OFF, sK0 = sb + L::K_OFF, sV0 = sb + L::V_OFF;
  int* pstart = reinterpret_cast<int*>(sm + L::PSTART_OFF);
  int2* pinfo = reinterpret_cast<int2*>(sm + L::PINFO_OFF);
  int* flags = reinterpret_cast<int*>(sm + L::FLAG_OFF);
  unsigned long long* turns = reinterpret_cast<unsigned long long*>(sm + L::TURNS_OFF);
  const uint32_t bar0 = sb + L::BAR_OFF;
  auto BAR = [&](int i) { return bar0 + 8u * uint32_t(i); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::MISC_OFF + 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(BAR(B_K_FULL + s), 1);
      mbar_init(BAR(B_K_READY + s), 128);
      mbar_init(BAR(B_K_FREE + s), 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(BAR(B_V_FULL + s), 1);
      mbar_init(BAR(B_V_FREE + s), 1);
    }
    for (int i = 0; i < kQT; ++i) {
      mbar_init(BAR(B_S_FULL + i), 1);
      mbar_init(BAR(B_P_FULL + i), KH ? 256 : 128);  // key halves: both warpgroups write P
    }
    mbar_init(BAR(B_Q_READY), 2 * 128);
    mbar_init(BAR(B_FINAL), 1);
    mbar_init(BAR(B_PV_DONE), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if constexpr (kRotate)
    for (int i = threadIdx.x; i < D / 2; i += blockDim.x) turns[i] = a.pos.turns[i];
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_u32(tmem_slot))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 2 * 4) {
    // ============================ Q preparation, softmax and epilogue of Q tile qt
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(Regs<kRotate, KH>::softmax));
    // qt: the warpgroup's Q tile, or (KH) its half of the keys of the one Q tile
    const int qt = warp >> 2;
    const int r = threadIdx.x & (kM - 1);  // row of the tile = TMEM lane
    const int token = tok0 + (KH ? 0 : qt * tpt) + r / G;
    const int h = g * G + r % G;
    const bool valid = token < Lq;
    const int m_row = valid ? mbase + token : -1;
    if (KH && qt == 1) {
      mbar_arrive(BAR(B_Q_READY));  // one Q tile, prepared by the first warpgroup
    } else {
      const uint32_t sQ = sQ0 + uint32_t(qt * L::QTILE);
      // The raw row is staged in this thread's own row of the Q tile (bf16, swizzled), then
      // rotated and scaled chunk by chunk in place, so a rotation partner at a run-time offset
      // (rotary_dim / 2) needs no register indexing.
      auto qaddr = [&](int k) { return sQ + uint32_t((k >> 3) * L::BLK) + swz(r, k & 7); };
      const uint4* src = reinterpret_cast<const uint4*>(a.q + ((size_t)(q0 + token) * a.Hq + h) * D);
#pragma unroll
      for (int k = 0; k < D / 8; ++k) st_shared_v4(qaddr(k), valid ? src[k] : make_uint4(0, 0, 0, 0));
      const float sc = a.pos.scale_log2;
      auto pack = [&](const float (&y)[8]) {
        if constexpr (kQkF16)
          return make_uint4(f2_to_h2(y[0] * sc, y[1] * sc), f2_to_h2(y[2] * sc, y[3] * sc),
                            f2_to_h2(y[4] * sc, y[5] * sc), f2_to_h2(y[6] * sc, y[7] * sc));
        else
          return make_uint4(f2_to_bf2(y[0] * sc, y[1] * sc), f2_to_bf2(y[2] * sc, y[3] * sc),
                            f2_to_bf2(y[4] * sc, y[5] * sc), f2_to_bf2(y[6] * sc, y[7] * sc));
      };
      auto unpack = [](uint4 u, float (&y)[8]) {
        y[0] = bf_lo(u.x); y[1] = bf_hi(u.x); y[2] = bf_lo(u.y); y[3] = bf_hi(u.y);
        y[4] = bf_lo(u.z); y[5] = bf_hi(u.z); y[6] = bf_lo(u.w); y[7] = bf_hi(u.w);
      };
      int done = 0;  // chunks [0, done) already written in their final form
      if constexpr (kRotate) {
        const uint32_t m = uint32_t(m_row < 0 ? 0 : m_row);
        const int rd = a.pos.rotary_dim, hr = rd / 2;
        const bool tab = a.pos.table != nullptr && int(m) < a.pos.max_pos;
        auto csf = [&](int i, float& sn, float& co) {
          if (tab) {
            co = a.pos.table[(size_t)m * rd + i];
            sn = a.pos.table[(size_t)m * rd + hr + i];
          } else {
            turn_sincos_fast(m, turns[i], sn, co);
          }
        };
        if (!a.pos.interleaved) {
#pragma unroll 1
          for (int c = 0; c < hr / 8; ++c) {  // chunk c against its partner c + hr/8
            float x1[8], x2[8];
            unpack(ld_shared_v4(qaddr(c)), x1);
            unpack(ld_shared_v4(qaddr(c + hr / 8)), x2);
            float y1[8], y2[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              float sn, co;
              csf(c * 8 + e, sn, co);
              y1[e] = x1[e] * co - x2[e] * sn;
              y2[e] = x1[e] * sn + x2[e] * co;
            }
            st_shared_v4(qaddr(c), pack(y1));
            st_shared_v4(qaddr(c + hr / 8), pack(y2));
          }
        } else {
#pragma unroll 1
          for (int k = 0; k < rd / 8; ++k) {  // adjacent pairs (2i, 2i+1), i = 4k .. 4k+3
            float x[8], y[8];
            unpack(ld_shared_v4(qaddr(k)), x);
#pragma unroll
            for (int w = 0; w < 4; ++w) {
              float sn, co;
              csf(k * 4 + w, sn, co);
              y[2 * w] = x[2 * w] * co - x[2 * w + 1] * sn;
              y[2 * w + 1] = x[2 * w] * sn + x[2 * w + 1] * co;
            }
            st_shared_v4(qaddr(k), pack(y));
          }
        }
        done = rd / 8;
      }
#pragma unroll 1
      for (int k = done; k < D / 8; ++k) {  // unrotated dimensions: scale and convert
        float x[8];
        unpack(ld_shared_v4(qaddr(k)), x);
        st_shared_v4(qaddr(k), pack(x));
      }
      fence_async_smem();
      mbar_arrive(BAR(B_Q_READY));
    }
    if (KH || qt < nq) {
      float slope = 0.f;
      if constexpr (POS == kAlibi) slope = a.pos.slopes[h] * 1.4426950408889634f;
      const uint32_t tl = tmem + (uint32_t(32 * (warp & 3)) << 16);
      const uint32_t tO = tl + uint32_t(2 * kN + qt * 128);
      float m_run = -INFINITY, l_run = 0.f;
      bool ok = true;
      for (int j = 0; j < ntiles; ++j) {
        const int slot = j % kSlots;
        const int buf = nq == 2 ? qt : (j & 1);  // S/P buffer and its barrier pair
        const uint32_t tS = tl + uint32_t(buf * kN);
        const bool got_s =
            wait_bar(BAR(B_S_FULL + buf), uint32_t(nq == 2 ? (j & 1) : ((j >> 1) & 1)), abort_flag, a.status);
        if (!__all_sync(0xffffffffu, got_s)) { ok = false; break; }
        tc_fence_after();
        const bool fast = flags[slot * 2] != 0;  // every key of the tile is visible to every row
        // this thread's scores in registers (the whole row, or with key halves its warpgroup's
        // 64 keys = page slots pg0 .. pg0 + 3): loads, one wait
        constexpr int NK = KH ? kN / 2 : kN, NPG = NK / kPage;
        const int pg0 = KH ? NPG * qt : 0;
        uint32_t v[NK];
#pragma unroll
        for (int c = 0; c < NK / 32; ++c)
          tmem_ld32(tS + uint32_t(pg0 * kPage + 32 * c), *reinterpret_cast<uint32_t(*)[32]>(v + 32 * c));
        tmem_wait_ld();
        // ALiBi bias -slope (m - p) for stage row t of a page, p = pstart + t: its per-key part
        // slope t goes onto the scores in packed pairs, its per-page part slope (pstart - m)
        // onto the page's maximum and into the page's exponent offset below (one packed FMA per
        // two scores instead of a multiply-add and an add per score)
        float bpg[NPG];
        if constexpr (POS == kAlibi) {
#pragma unroll
          for (int pp = 0; pp < NPG; ++pp) {
            bpg[pp] = slope * float(pstart[slot * kPagesPerTile + pg0 + pp] - m_row);
#pragma unroll
            for (int t = 0; t < kPage; t += 2) {
              float2 x = make_float2(__uint_as_float(v[pp * kPage + t]), __uint_as_float(v[pp * kPage + t + 1]));
              x = __ffma2_rn(make_float2(slope, slope), make_float2(float(t), float(t + 1)), x);
              v[pp * kPage + t] = __float_as_uint(x.x);
              v[pp * kPage + t + 1] = __float_as_uint(x.y);
            }
          }
        }
        if (!fast) {  // stage row t of a page holds key p = pstart + t; visible iff t >= lo, p <= m
#pragma unroll
          for (int pp = 0; pp < NPG; ++pp) {
            const int st = pstart[slot * kPagesPerTile + pg0 + pp];
            const int lo = pinfo[slot * kPagesPerTile + pg0 + pp].y;
            const int hi = m_row - st + 1;
#pragma unroll
            for (int t = 0; t < kPage; ++t)
              if (!(t >= lo && t < hi)) v[pp * kPage + t] = __float_as_uint(-INFINITY);
          }
        }
        // row max over the scores: independent runs of three-input maxima over each page's 16,
        // then a tree
        float mq[NPG];
#pragma unroll
        for (int q = 0; q < NPG; ++q) {
          const float* x = reinterpret_cast<const float*>(v + 16 * q);
          float m = max3f(x[0], x[1], x[2]);
#pragma unroll
          for (int e = 3; e < 15; e += 2) m = max3f(m, x[e], x[e + 1]);
          mq[q] = fmaxf(m, x[15]);
          if constexpr (POS == kAlibi) mq[q] += bpg[q];
        }
        float mx;
        if constexpr (KH)
          mx = max3f(max3f(mq[0], mq[1], mq[2]), mq[3], mq[3]);
        else
          mx = max3f(max3f(mq[0], mq[1], mq[2]), max3f(mq[3], mq[4], mq[5]), fmaxf(mq[6], mq[7]));
        const bool need = mx > m_run + kTau;
        const float m_new = need ? mx : m_run;
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;  // fully masked row: every p is 0
        float2 mneg[NPG];  // exponent offset per page: -m, with ALiBi the page's bias part too
#pragma unroll
        for (int pp = 0; pp < NPG; ++pp) {
          const float o = POS == kAlibi ? bpg[pp] - m_use : -m_use;
          mneg[pp] = make_float2(o, o);
        }
        float2 sum4[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                          make_float2(0.f, 0.f)};  // four independent partial sums
        // P packed to bf16 pairs in place: pair e (keys 2e, 2e+1) lands in v[e] (already consumed)
#pragma unroll
        for (int e = 0; e < NK / 2; ++e) {
          float2 x = make_float2(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1]));
          x = __fadd2_rn(x, mneg[e / (kPage / 2)]);
          const float2 ev = make_float2(ex2(x.x), ex2(x.y));
          sum4[e & 3] = __fadd2_rn(sum4[e & 3], ev);
          v[e] = f2_to_bf2(ev.x, ev.y);
        }
        const float2 s01 = __fadd2_rn(sum4[0], sum4[1]), s23 = __fadd2_rn(sum4[2], sum4[3]);
        const float2 s03 = __fadd2_rn(s01, s23);
        const float sum = s03.x + s03.y;
        const float alpha = (j > 0 && need && m_run != -INFINITY) ? ex2(m_run - m_new) : 1.f;
        l_run = (j == 0) ? sum : l_run * alpha + sum;
        // O rescale needs the previous tile's PV complete: with two Q tiles the S commit waited
        // for covers it; with one, S of tile j was issued before PV of tile j-1, so wait for it
        if (nq == 1 && j > 0) {
          const bool got_pv = wait_bar(BAR(B_PV_DONE), uint32_t((j - 1) & 1), abort_flag, a.status);
          if (!__all_sync(0xffffffffu, got_pv)) { ok = false; break; }
          tc_fence_after();
        }
        if (__any_sync(0xffffffffu, j > 0 && alpha != 1.f)) {
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tO + uint32_t(c * 32), o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(tO + uint32_t(c * 32), o);
          }
        }
        m_run = m_new;
        // P row -> TMEM over the first 64 columns of S (column e holds keys 2e, 2e+1); with key
        // halves each warpgroup writes its 32 columns over the start of its own S columns
        // (keys 64h .. 64h + 63 -> columns 64h .. 64h + 31), never over the other's scores
#pragma unroll
        for (int c = 0; c < NK / 64; ++c)
          tmem_st32(tS + uint32_t(pg0 * kPage + 32 * c), *reinterpret_cast<const uint32_t(*)[32]>(v + 32 * c));
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(BAR(B_P_FULL + buf));
      }
      const bool got_last = ok && wait_bar(BAR(B_FINAL), 0, abort_flag, a.status);
      if constexpr (KH) {
        // The two key halves of a row are two partial softmaxes (O_A over keys 0-63 of every
        // tile, O_B over keys 64-127): merged by their maxima and sums, exchanged through the
        // unused second Q tile's space.  Each warpgroup writes its 64 output columns.
        float2* xml = reinterpret_cast<float2*>(sm + L::Q_OFF + L::QTILE);
        xml[qt * kM + r] = make_float2(l_run > 0.f ? m_run : -INFINITY, l_run);
        named_sync(1, 2 * kM);  // the two softmax warpgroups
        const float2 mine = xml[qt * kM + r], other = xml[(qt ^ 1) * kM + r];
        const float2 hA = qt == 0 ? mine : other, hB = qt == 0 ? other : mine;
        const float M = fmaxf(hA.x, hB.x);
        const float wA = hA.y > 0.f ? ex2(hA.x - M) : 0.f, wB = hB.y > 0.f ? ex2(hB.x - M) : 0.f;
        const float Lt = wA * hA.y + wB * hB.y;
        if (__all_sync(0xffffffffu, got_last)) {
          tc_fence_after();
          const bool part = a.S > 1;
          const float inv = part ? 1.f : (Lt > 0.f ? 1.f / Lt : 0.f);
          const size_t pi = ((size_t)(q0 + token) * a.Hq + h) * a.S + split;
          __nv_bfloat16* orow = a.out + ((size_t)(q0 + token) * a.Hq + h) * D;
#pragma unroll 1
          for (int c = 0; c < D / 64; ++c) {
            const int col = qt * (D / 2) + c * 32;
            uint32_t oa[32], ob[32];
            tmem_ld32(tl + uint32_t(2 * kN + col), oa);
            tmem_ld32(tl + uint32_t(3 * kN + col), ob);
            tmem_wait_ld();
            float o[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = (wA * __uint_as_float(oa[e]) + wB * __uint_as_float(ob[e])) * inv;
            if (valid && part) {
              float4* dst = reinterpret_cast<float4*>(a.part_o + pi * D + col);
#pragma unroll
              for (int q4 = 0; q4 < 8; ++q4) dst[q4] = make_float4(o[4 * q4], o[4 * q4 + 1], o[4 * q4 + 2], o[4 * q4 + 3]);
            } else if (valid) {
              uint4* dst = reinterpret_cast<uint4*>(orow + col);
#pragma unroll
              for (int q4 = 0; q4 < 4; ++q4)
                dst[q4] = make_uint4(f2_to_bf2(o[8 * q4], o[8 * q4 + 1]), f2_to_bf2(o[8 * q4 + 2], o[8 * q4 + 3]),
                                     f2_to_bf2(o[8 * q4 + 4], o[8 * q4 + 5]), f2_to_bf2(o[8 * q4 + 6], o[8 * q4 + 7]));
            }
          }
          if (valid && qt == 0) {
            if (part) {
              a.part_ml[pi * 2] = Lt > 0.f ? M : -INFINITY;
              a.part_ml[pi * 2 + 1] = Lt;
            } else if (a.lse) {
              a.lse[(size_t)(q0 + token) * a.Hq + h] = (M + log2f(Lt)) * 0.6931471805599453f;
            }
          }
        }
      } else if (__all_sync(0xffffffffu, got_last) && a.S > 1) {
        tc_fence_after();
        const size_t pi = ((size_t)(q0 + token) * a.Hq + h) * a.S + split;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tO + uint32_t(c * 32), o);
          tmem_wait_ld();
          if (valid) {
            float4* dst = reinterpret_cast<float4*>(a.part_o + pi * D + c * 32);
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4)
              dst[q4] = make_float4(__uint_as_float(o[q4 * 4]), __uint_as_float(o[q4 * 4 + 1]),
                                    __uint_as_float(o[q4 * 4 + 2]), __uint_as_float(o[q4 * 4 + 3]));
          }
        }
        if (valid) {
          a.part_ml[pi * 2] = l_run > 0.f ? m_run : -INFINITY;
          a.part_ml[pi * 2 + 1] = l_run;
        }
      } else if (__all_sync(0xffffffffu, got_last)) {
        tc_fence_after();
        const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
        __nv_bfloat16* orow = a.out + ((size_t)(q0 + token) * a.Hq + h) * D;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tO + uint32_t(c * 32), o);
          tmem_wait_ld();
          if (valid) {
            uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4)
              dst[q4] = make_uint4(f2_to_bf2(__uint_as_float(o[q4 * 8 + 0]) * inv, __uint_as_float(o[q4 * 8 + 1]) * inv),
                                   f2_to_bf2(__uint_as_float(o[q4 * 8 + 2]) * inv, __uint_as_float(o[q4 * 8 + 3]) * inv),
                                   f2_to_bf2(__uint_as_float(o[q4 * 8 + 4]) * inv, __uint_as_float(o[q4 * 8 + 5]) * inv),
                                   f2_to_bf2(__uint_as_float(o[q4 * 8 + 6]) * inv, __uint_as_float(o[q4 * 8 + 7]) * inv));
          }
        }
        if (valid && a.lse) a.lse[(size_t)(q0 + token) * a.Hq + h] = (m_run + log2f(l_run)) * 0.6931471805599453f;
      }
    }
  } else if (warp < kProdWarp) {
    // ============================ K rotation
    // Thread rt works on page slot ps = rt / 16 of every tile.  Full half-split rotation: it owns
    // chunk pair c (dims 8c..8c+7 and their partners 8c+D/2..) for NCP rows of the page and keeps
    // the cos/sin of those 8 frequencies in registers, recomputed only when its page slot's
    // Delta changes (pages inside one document share it), so there is no cos/sin buffer and no
    // barrier among the rotation threads.  Partial rotary_dim / interleaved pairs: each thread
    // owns one chunk task (a rotated chunk pair or chunk, or one unrotated chunk converted to
    // f16) for all 16 rows of its page.
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(Regs<kRotate, KH>::rot));
    const int rt = threadIdx.x - kRotWarp0 * 32;
    const int ps = rt / kPage, l = rt % kPage;
    constexpr int NCP = D / 16;  // chunk pairs per row (full width)
    bool ok = true;              // once a wait gives up, the thread skips work but keeps arriving
    float co[8], sn[8];
    int cur_delta = -1;
    // this thread's task in the generic layout: rotated chunk pair / chunk (kind 0 / 1) or tail
    // chunk converted to f16 (kind 2), or nothing (kind 3)
    int g_kind = 3, g_chunk = 0, g_part = 0, g_f0 = 0;
    if constexpr (POS == kRopeX) {
      const int rd = a.pos.rotary_dim;
      const int nrot = a.pos.interleaved ? rd / 8 : rd / 16, ntail = (D - rd) / 8;
      if (l < nrot) {
        g_kind = a.pos.interleaved ? 1 : 0;
        g_chunk = l;
        g_part = l + rd / 16;                  // half-split partner chunk
        g_f0 = a.pos.interleaved ? 4 * l : 8 * l;  // first frequency of the task
      } else if (l < nrot + ntail) {
        g_kind = 2;
        g_chunk = rd / 8 + (l - nrot);
      }
    }
    for (int j = 0; j < ntiles; ++j) {
      const int s = j % kKStages, slot = j % kSlots;
      if (ok) ok = wait_bar(BAR(B_K_FULL + s), uint32_t((j / kKStages) & 1), abort_flag, a.status);
      if constexpr (kRotate) {
        const int2 pi = ok ? pinfo[slot * kPagesPerTile + ps] : make_int2(0, kPage);  // {Delta, lo}
        const uint32_t sK = sK0 + uint32_t(s * L::TILE);
        if (pi.y < kPage) {  // the page holds keys (rows before lo are zeros)
          if constexpr (POS == kRope) {
            const int c = l % NCP, g = l / NCP;
            if (pi.x != cur_delta) {
              cur_delta = pi.x;
#pragma unroll
              for (int e = 0; e < 8; ++e) turn_sincos_fast(uint32_t(pi.x), turns[8 * c + e], sn[e], co[e]);
            }
#pragma unroll
            for (int i = 0; i < NCP; ++i) {
              const int t = g * NCP + i;
              if (t < pi.y) continue;
              const int r = ps * kPage + t;  // row of the tile
              // element 8c + e and its partner 8c + e + D/2: the same chunk slot of the other
              // column block (D = 128) or chunk c + 4 of the same block (D = 64)
              const uint32_t a1 = sK + swz(r, c);
              const uint32_t a2 = (D == 128) ? sK + uint32_t(L::BLK) + swz(r, c) : sK + swz(r, c + 4);
              uint4 u1 = ld_shared_v4(a1), u2 = ld_shared_v4(a2);
              uint32_t* p1 = reinterpret_cast<uint32_t*>(&u1);
              uint32_t* p2 = reinterpret_cast<uint32_t*>(&u2);
#pragma unroll
              for (int w = 0; w < 4; ++w) {
                const float2 cv = make_float2(co[2 * w], co[2 * w + 1]), sv = make_float2(sn[2 * w], sn[2 * w + 1]);
                const float2 x1 = bf2_to_f2(p1[w]), x2 = bf2_to_f2(p2[w]);
                const float2 t1 = __fmul2_rn(x2, sv), t2 = __fmul2_rn(x2, cv);
                const float2 y1 = __ffma2_rn(x1, cv, make_float2(-t1.x, -t1.y));  // x1 c - x2 s
                const float2 y2 = __ffma2_rn(x1, sv, t2);                          // x1 s + x2 c
                p1[w] = f2_to_h2(y1.x, y1.y);
                p2[w] = f2_to_h2(y2.x, y2.y);
              }
              st_shared_v4(a1, u1);
              st_shared_v4(a2, u2);
            }
          } else {  // POS == kRopeX
            auto kaddr = [&](int r, int k) { return sK + uint32_t((k >> 3) * L::BLK) + swz(r, k & 7); };
            if (g_kind < 2 && pi.x != cur_delta) {
              cur_delta = pi.x;
              const int nf = g_kind == 0 ? 8 : 4;
#pragma unroll
              for (int e = 0; e < 8; ++e)
                if (e < nf) turn_sincos_fast(uint32_t(pi.x), turns[g_f0 + e], sn[e], co[e]);
            }
#pragma unroll 1
            for (int t = pi.y; t < kPage && g_kind < 3; ++t) {
              const int r = ps * kPage + t;
              if (g_kind == 0) {  // half-split pairs: chunk against its partner chunk + rotary_dim/16
                const uint32_t a1 = kaddr(r, g_chunk), a2 = kaddr(r, g_part);
                uint4 u1 = ld_shared_v4(a1), u2 = ld_shared_v4(a2);
                uint32_t* p1 = reinterpret_cast<uint32_t*>(&u1);
                uint32_t* p2 = reinterpret_cast<uint32_t*>(&u2);
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                  const float2 x1 = bf2_to_f2(p1[w]), x2 = bf2_to_f2(p2[w]);
                  p1[w] = f2_to_h2(x1.x * co[2 * w] - x2.x * sn[2 * w], x1.y * co[2 * w + 1] - x2.y * sn[2 * w + 1]);
                  p2[w] = f2_to_h2(x1.x * sn[2 * w] + x2.x * co[2 * w], x1.y * sn[2 * w + 1] + x2.y * co[2 * w + 1]);
                }
                st_shared_v4(a1, u1);
                st_shared_v4(a2, u2);
              } else if (g_kind == 1) {  // adjacent pairs (x_2i, x_2i+1), i = 4 chunk + w
                const uint32_t a1 = kaddr(r, g_chunk);
                uint4 u = ld_shared_v4(a1);
                uint32_t* pw = reinterpret_cast<uint32_t*>(&u);
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                  const float x0 = bf_lo(pw[w]), x1 = bf_hi(pw[w]);
                  pw[w] = f2_to_h2(x0 * co[w] - x1 * sn[w], x0 * sn[w] + x1 * co[w]);
                }
                st_shared_v4(a1, u);
              } else {  // unrotated tail: bf16 -> f16 (QK^T has one operand type)
                const uint32_t a1 = kaddr(r, g_chunk);
                uint4 u = ld_shared_v4(a1);
                uint32_t* pw = reinterpret_cast<uint32_t*>(&u);
#pragma unroll
                for (int w = 0; w < 4; ++w) pw[w] = f2_to_h2(bf_lo(pw[w]), bf_hi(pw[w]));
                st_shared_v4(a1, u);
              }
            }
          }
        }
        fence_async_smem();
      }
      mbar_arrive(BAR(B_K_READY + s));
    }
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(Regs<kRotate, KH>::issue));
    if (warp == kProdWarp) {
      // ============================ block words + TMA
      // Issue order K0, K1, V0, K2, V1, ...: a K stage is refilled once both its QK^T are done, a
      // V stage once both its PV are done, and no K load waits behind an earlier tile's PV.
      const uint64_t* mrow = a.meta + (size_t)b * a.max_blocks;
      int* pgid = reinterpret_cast<int*>(sm + L::PGID_OFF);
      // With ALiBi the bias grows towards the query, so the newest keys hold each row's maximum:
      // visiting the tiles newest first fixes the running max at once and the O rescale of the
      // lazy softmax (only when a max grows by more than 8) almost never runs.  Softmax is
      // indifferent to key order, and every per-tile fact travels with the tile's slot.
      auto tile_of = [&](int j) { return POS == kAlibi ? t0 + ntiles - 1 - j : t0 + j; };
      auto fetch = [&](int j) -> uint64_t {  // lane < 8: block word of page slot `lane` of tile j
        const int jb = tile_of(j) * kPagesPerTile + lane;
        return (lane < kPagesPerTile && j < ntiles && jb < nb) ? ldg_u64(mrow + jb) : 0ull;
      };
      uint64_t w_next = fetch(0);
      int issued_k = 0, issued_v = 0;
      // K of tile j: wait for its stage, publish the tile's metadata, load the pages
      auto issue_k = [&](int j) -> bool {
        const int s = j % kKStages, slot = j % kSlots;
        const uint64_t w = w_next;
        w_next = fetch(j + 1);  // prefetch: its latency overlaps this tile's waits
        // rows: keys of the page that some row of this CTA may see.  Only a document's last page
        // is partial (a prefix of n_valid rows); in the query segment the rows past the CTA's
        // last token m_max are not needed (and may not be written yet).
        int rows = 0, start = 0, page = 0, delta = 0;
        const int jb = tile_of(j) * kPagesPerTile + lane;
        if (lane < kPagesPerTile && jb < nb) {
          page = int(word_page(w));
          delta = int(word_delta(w));
          start = delta + kPage * int(word_pg(w));
          rows = max(0, min(min(int(word_nvalid(w)), kPage), m_max - start + 1));
          if (page >= a.num_pages) {
            set_status(a.status, LAZY_STATUS_BAD_PAGE);
            rows = 0;
          }
        }
        const int lo = kPage - rows;  // the page is loaded from row -lo: stage rows [lo, 16) hold its keys
        if (j >= kKStages) {
          const bool freed = wait_bar(BAR(B_K_FREE + s), uint32_t(((j / kKStages) - 1) & 1), abort_flag, a.status);
          if (!__all_sync(0xffffffffu, freed)) return false;
        }
        const int zc = page * a.Hkv + g;  // page-head coordinate of the tensor map
        if (lane < kPagesPerTile) {
          pinfo[slot * kPagesPerTile + lane] = make_int2(delta, lo);
          pgid[slot * kPagesPerTile + lane] = rows > 0 ? zc : -1;
          pstart[slot * kPagesPerTile + lane] = start - lo;
        }
        const int all16 = __all_sync(0xffffffffu, lane >= kPagesPerTile || rows == kPage);
        const int last_start = __shfl_sync(0xffffffffu, start, kPagesPerTile - 1);
        if (lane == 0) flags[slot * 2] = all16 && (last_start + kPage - 1 <= m_min);  // every key visible to every row
        __syncwarp();
        const uint32_t loaded = __ballot_sync(0xffffffffu, lane < kPagesPerTile && rows > 0);
        const uint32_t bytes = uint32_t(__popc(loaded)) * kPage * D * 2;  // whole boxes, zero rows included
        const uint32_t sK = sK0 + uint32_t(s * L::TILE);
        if (lane == 0) mbar_arrive_expect_tx(BAR(B_K_FULL + s), bytes);
        __syncwarp();
        if (lane < kPagesPerTile && rows > 0)  // one lane per page: TMA issue is per-instruction bound
#pragma unroll
          for (int cb = 0; cb < L::CB; ++cb)
            tma_load_3d(sK + uint32_t(cb * L::BLK + lane * kPage * 128), &tmk, cb * 64, -lo, zc, BAR(B_K_FULL + s));
        __syncwarp();
        issued_k = j + 1;
        return true;
      };
      // V of tile j (its metadata was published with its K).  A page slot past the CTA's last
      // block gets no load; its stage rows still meet the PV MMA (with zero weights), so they are
      // cleared here, after the stage's previous PV is done, instead of keeping stale bits.
      auto issue_v = [&](int j) -> bool {
        const int s = j % kVStages, slot = j % kSlots;
        if (j >= kVStages) {
          const bool freed = wait_bar(BAR(B_V_FREE + s), uint32_t(((j / kVStages) - 1) & 1), abort_flag, a.status);
          if (!__all_sync(0xffffffffu, freed)) return false;
        }
        const uint32_t sV = sV0 + uint32_t(s * L::TILE);
        const int zc = lane < kPagesPerTile ? pgid[slot * kPagesPerTile + lane] : -1;
        const int lo = lane < kPagesPerTile ? pinfo[slot * kPagesPerTile + lane].y : kPage;
        const uint32_t loaded = __ballot_sync(0xffffffffu, zc >= 0);
        const uint32_t empty = ~loaded & ((1u << kPagesPerTile) - 1u);
        if (empty) {  // a warp-wide store of 16 B per lane covers two rows of a column block
          for (int pp = 0; pp < kPagesPerTile; ++pp) {
            if (!((empty >> pp) & 1u)) continue;
#pragma unroll
            for (int cb = 0; cb < L::CB; ++cb)
#pragma unroll
              for (int i = 0; i < kPage * 8 / 32; ++i) {
                const int row = pp * kPage + (i * 32 + lane) / 8, c = (i * 32 + lane) % 8;
                st_shared_v4(sV + uint32_t(cb * L::BLK) + swz(row, c), make_uint4(0, 0, 0, 0));
              }
          }
          fence_async_smem();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive_expect_tx(BAR(B_V_FULL + s), uint32_t(__popc(loaded)) * kPage * D * 2);
        __syncwarp();
        if (zc >= 0)
#pragma unroll
          for (int cb = 0; cb < L::CB; ++cb)
            tma_load_3d(sV + uint32_t(cb * L::BLK + lane * kPage * 128), &tmv, cb * 64, -lo, zc, BAR(B_V_FULL + s));
        __syncwarp();
        issued_v = j + 1;
        return true;
      };
      // K runs kKStages - 1 tiles ahead of V: K0 K1 K2 V0 K3 V1 ...
      bool ok = true;
      const bool own_v = !(SPLIT_V && nq == 1);  // otherwise warp 14 issues V
      for (int j = 0; j < kKStages - 1 && j < ntiles && ok; ++j) ok = issue_k(j);
      for (int j = 0; j < ntiles && ok; ++j) {
        if (j + kKStages - 1 < ntiles) ok = issue_k(j + kKStages - 1);
        if (ok && own_v) ok = issue_v(j);
      }
      // never leave copies in flight: wait (bounded) for the last loads of every stage
      if (lane == 0) {
        for (int j = max(0, issued_k - kKStages); j < issued_k; ++j) {
          const uint32_t bar = BAR(B_K_FULL + j % kKStages), par = uint32_t((j / kKStages) & 1);
          WaitClock clk;
          while (!mbar_test(bar, par) && !clk.expired()) {
          }
        }
        for (int j = max(0, issued_v - kVStages); j < issued_v; ++j) {
          const uint32_t bar = BAR(B_V_FULL + j % kVStages), par = uint32_t((j / kVStages) & 1);
          WaitClock clk;
          while (!mbar_test(bar, par) && !clk.expired()) {
          }
        }
      }
    } else if (SPLIT_V && warp == kVProdWarp && nq == 1) {
      // ============================ V producer (one live Q tile)
      // V's own producer (SPLIT_V): it reads the block words itself; pages, rows and zero fill
      // follow the K producer's rules, and issue_v's stage protocol.
      const uint64_t* mrow = a.meta + (size_t)b * a.max_blocks;
      auto tile_of = [&](int j) { return POS == kAlibi ? t0 + ntiles - 1 - j : t0 + j; };
      auto fetch = [&](int j) -> uint64_t {
        const int jb = tile_of(j) * kPagesPerTile + lane;
        return (lane < kPagesPerTile && j < ntiles && jb < nb) ? ldg_u64(mrow + jb) : 0ull;
      };
      uint64_t w_next = fetch(0);
      int issued_v = 0;
      // With rotation, V waits until Q is ready (V is first needed by PV(0), after QK(0) and its
      // softmax): the K chain, whose tiles must also be rotated, has the copy engine to itself
      // while the Q rows are prepared.  Measured: 322 -> 308 us on a 32-request, 12 000-key
      // YaRN prefill, and slower for the ALiBi decode, which keeps the early V copies.
      int ntiles_v = ntiles;
      if constexpr (kRotate) {
        const bool q_ready = wait_bar(BAR(B_Q_READY), 0, abort_flag, a.status);
        if (!__all_sync(0xffffffffu, q_ready)) ntiles_v = 0;
      }
      for (int j = 0; j < ntiles_v; ++j) {
        const int s = j % kVStages;
        const uint64_t w = w_next;
        w_next = fetch(j + 1);
        int rows = 0, zc = 0;
        const int jb = tile_of(j) * kPagesPerTile + lane;
        if (lane < kPagesPerTile && jb < nb) {
          const int page = int(word_page(w));
          const int start = int(word_delta(w)) + kPage * int(word_pg(w));
          rows = max(0, min(min(int(word_nvalid(w)), kPage), m_max - start + 1));
          if (page >= a.num_pages) rows = 0;  // reported by the K producer
          zc = page * a.Hkv + g;
        }
        const int lo = kPage - rows;
        if (j >= kVStages) {
          const bool freed = wait_bar(BAR(B_V_FREE + s), uint32_t(((j / kVStages) - 1) & 1), abort_flag, a.status);
          if (!__all_sync(0xffffffffu, freed)) break;
        }
        const uint32_t sV = sV0 + uint32_t(s * L::TILE);
        const uint32_t loaded = __ballot_sync(0xffffffffu, lane < kPagesPerTile && rows > 0);
        const uint32_t empty = ~loaded & ((1u << kPagesPerTile) - 1u);
        if (empty) {  // page slots past the last block: cleared (they meet PV with zero weights)
          for (int pp = 0; pp < kPagesPerTile; ++pp) {
            if (!((empty >> pp) & 1u)) continue;
#pragma unroll
            for (int cb = 0; cb < L::CB; ++cb)
#pragma unroll
              for (int i = 0; i < kPage * 8 / 32; ++i) {
                const int row = pp * kPage + (i * 32 + lane) / 8, c = (i * 32 + lane) % 8;
                st_shared_v4(sV + uint32_t(cb * L::BLK) + swz(row, c), make_uint4(0, 0, 0, 0));
              }
          }
          fence_async_smem();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive_expect_tx(BAR(B_V_FULL + s), uint32_t(__popc(loaded)) * kPage * D * 2);
        __syncwarp();
        if (lane < kPagesPerTile && rows > 0)
#pragma unroll
          for (int cb = 0; cb < L::CB; ++cb)
            tma_load_3d(sV + uint32_t(cb * L::BLK + lane * kPage * 128), &tmv, cb * 64, -lo, zc, BAR(B_V_FULL + s));
        __syncwarp();
        issued_v = j + 1;
      }
      if (lane == 0)  // never leave copies in flight
        for (int j = max(0, issued_v - kVStages); j < issued_v; ++j) {
          const uint32_t bar = BAR(B_V_FULL + j % kVStages), par = uint32_t((j / kVStages) & 1);
          WaitClock clk;
          while (!mbar_test(bar, par) && !clk.expired()) {
          }
        }
    } else if (warp == kMmaWarp) {
      // ============================ MMA issue (one thread)
      if (lane == 0) {
        constexpr uint32_t IQK = idesc_mma(kM, kN, 0, kQkF16 ? 1 : 0);
        constexpr uint32_t IPV = idesc_mma(kM, D, 1, 0);
        bool ok = wait_bar(BAR(B_Q_READY), 0, abort_flag, a.status);
        auto qk = [&](int qt, int j) {  // S_qt = Q_qt K_j^T
          const uint32_t sK = sK0 + uint32_t((j % kKStages) * L::TILE), sQ = sQ0 + uint32_t(qt * L::QTILE);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = uint32_t((kk >> 2) * L::BLK + (kk & 3) * 32);
            mma_bf16(tmem + uint32_t(qt * kN), sdesc(sQ + off, 16, 1024), sdesc(sK + off, 16, 1024), IQK,
                     kk > 0 ? 1u : 0u);
          }
          mma_commit(BAR(B_S_FULL + qt));
        };
        auto pv = [&](int qt, int jj) {  // O_qt += P_qt V_jj, P from TMEM (8 columns per 16 keys)
          const uint32_t sV = sV0 + uint32_t((jj % kVStages) * L::TILE);
#pragma unroll
          for (int kk = 0; kk < kN / 16; ++kk)
            mma_ts(tmem + uint32_t(2 * kN + qt * 128), tmem + uint32_t(qt * kN + kk * 8),
                   sdesc(sV + uint32_t(kk * 16 * 128), L::BLK, 1024), IPV, (jj > 0 || kk > 0) ? 1u : 0u);
        };
        auto wait_v = [&](int jj) -> bool {  // every V_FULL phase of both stages, in tile order
          return wait_bar(BAR(B_V_FULL + jj % kVStages), uint32_t((jj / kVStages) & 1), abort_flag, a.status);
        };
        if (nq == 1) {
          // one live Q tile: tile j's scores in S_{j%2}; order QK(0) QK(1) | PV(0) QK(2) | PV(1) ...
          auto qk1 = [&](int j) -> bool {
            if (!wait_bar(BAR(B_K_READY + j % kKStages), uint32_t((j / kKStages) & 1), abort_flag, a.status))
              return false;
            tc_fence_after();
            const uint32_t sK = sK0 + uint32_t((j % kKStages) * L::TILE);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = uint32_t((kk >> 2) * L::BLK + (kk & 3) * 32);
              mma_bf16(tmem + uint32_t((j & 1) * kN), sdesc(sQ0 + off, 16, 1024), sdesc(sK + off, 16, 1024), IQK,
                       kk > 0 ? 1u : 0u);
            }
            mma_commit(BAR(B_S_FULL + (j & 1)));
            mma_commit(BAR(B_K_FREE + j % kKStages));
            return true;
          };
          if (ok) ok = qk1(0);
          if (ok && ntiles > 1) ok = qk1(1);
          for (int j = 0; j < ntiles && ok; ++j) {
            ok = wait_bar(BAR(B_P_FULL + (j & 1)), uint32_t((j >> 1) & 1), abort_flag, a.status) &&
                 wait_v(j);
            if (!ok) break;
            tc_fence_after();
            const uint32_t sV = sV0 + uint32_t((j % kVStages) * L::TILE);
#pragma unroll
            for (int kk = 0; kk < kN / 16; ++kk) {
              // key halves: keys 0-63 into O_A (columns 2 kN), keys 64-127 into O_B (3 kN), each
              // half's P at the start of its own S columns
              const int hk = KH ? kk / 4 : 0;
              const uint32_t pcol = uint32_t((j & 1) * kN + (KH ? 64 * hk + (kk % 4) * 8 : kk * 8));
              mma_ts(tmem + uint32_t((2 + hk) * kN), tmem + pcol, sdesc(sV + uint32_t(kk * 16 * 128), L::BLK, 1024),
                     IPV, (j > 0 || kk > (KH ? 4 * hk : 0)) ? 1u : 0u);
            }
            mma_commit(BAR(B_PV_DONE));
            mma_commit(BAR(B_V_FREE + j % kVStages));
            if (j + 2 < ntiles) ok = qk1(j + 2);
          }
          ok = false;  // the two-tile schedule below is skipped
        }
        if (ok) ok = wait_bar(BAR(B_K_READY), 0, abort_flag, a.status);
        if (ok) {
          tc_fence_after();
          qk(0, 0);
          if (nq == 2) qk(1, 0);
          mma_commit(BAR(B_K_FREE));
        }
        for (int j = 1; j < ntiles && ok; ++j) {
          const int s = j % kKStages, sp = (j - 1) % kVStages;
          if (!wait_bar(BAR(B_P_FULL), uint32_t((j - 1) & 1), abort_flag, a.status) || !wait_v(j - 1)) {
            ok = false;
            break;
          }
          tc_fence_after();
          pv(0, j - 1);
          if (!wait_bar(BAR(B_K_READY + s), uint32_t((j / kKStages) & 1), abort_flag, a.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          qk(0, j);
          if (nq == 2) {
            if (!wait_bar(BAR(B_P_FULL + 1), uint32_t((j - 1) & 1), abort_flag, a.status)) {
              ok = false;
              break;
            }
            tc_fence_after();
            pv(1, j - 1);
          }
          mma_commit(BAR(B_V_FREE + sp));
          if (nq == 2) qk(1, j);
          mma_commit(BAR(B_K_FREE + s));
        }
        if (ok) {
          const int jl = ntiles - 1;
          ok = wait_bar(BAR(B_P_FULL), uint32_t(jl & 1), abort_flag, a.status) && wait_v(jl);
          if (ok) {
            tc_fence_after();
            pv(0, jl);
          }
          if (ok && nq == 2) {
            ok = wait_bar(BAR(B_P_FULL + 1), uint32_t(jl & 1), abort_flag, a.status);
            if (ok) {
              tc_fence_after();
              pv(1, jl);
            }
          }
          if (ok) mma_commit(BAR(B_V_FREE + jl % kVStages));
        }
        // every MMA must be complete before TMEM is released (and before the epilogue reads O)
        mma_commit(BAR(B_FINAL));
        WaitClock clk;
        while (!mbar_test(BAR(B_FINAL), 0) && !clk.expired()) {
        }
      }
      __syncwarp();
    }
  }

  pdl_trigger();  // every CTA of the grid is running once all have reached this point
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem) : "memory");
  }
}

}  // namespace tc

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encoder() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// Tensor map of a paged cache as a 3-D tensor: columns (D, bf16) x rows of a page (16) x
// page-heads (num_pages * Hkv).  One TMA box = 64 columns x 16 rows x 1 page-head with the
// 128-byte swizzle.  Rows outside [0, 16) of a page are outside the tensor and read as zero
// (FLOAT_OOB_FILL_NONE), so a box started at a negative row zero-fills the rows before row 0.
static int cache_map(CUtensorMap* map, const void* base, int num_pages, int Hkv, int D) {
  EncodeTiledFn enc = encoder();
  if (!enc) return fail(LAZY_ECUDA, "cuTensorMapEncodeTiled is unavailable");
  const cuuint64_t dims[3] = {cuuint64_t(D), cuuint64_t(kPage), cuuint64_t(num_pages) * cuuint64_t(Hkv)};
  const cuuint64_t strides[2] = {cuuint64_t(D) * 2, cuuint64_t(kPage) * D * 2};
  const cuuint32_t box[3] = {64, kPage, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(LAZY_ECUDA, "cuTensorMapEncodeTiled failed (%d)", int(r));
  return LAZY_OK;
}

template <int D, int POS, bool SPLIT_V, bool KH>
static int launch_tc(const CUtensorMap& mk, const CUtensorMap& mv, const tc::Args& a, int max_q, cudaStream_t st) {
  // (decode mode: max_q = 1, one query row per request)
  using L = tc::Layout<D>;
  auto kern = tc::prefill_tc_kernel<D, POS, SPLIT_V, KH>;
  static bool attr[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (!attr[dev & 63]) {
    LAZY_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM));
    attr[dev & 63] = true;
  }
  // The warpgroups re-split the launch allocation with setmaxnreg; that split is only valid
  // (and a growing warpgroup only ever gets its registers) if the kernel launches with exactly
  // kRegsLaunch registers per thread.
  static int regs[64] = {};
  if (!regs[dev & 63]) {
    cudaFuncAttributes fa;
    LAZY_CUDA_TRY(cudaFuncGetAttributes(&fa, kern));
    regs[dev & 63] = fa.numRegs;
  }
  if (regs[dev & 63] != tc::kRegsLaunch)
    return fail(LAZY_ECUDA, "prefill kernel built with %d registers per thread, expected %d", regs[dev & 63],
                tc::kRegsLaunch);
  const int G = a.Hq / a.Hkv;
  const int rows_tok = tc::kQT * (tc::kM / G);  // tokens per CTA
  dim3 grid(unsigned((max_q + rows_tok - 1) / rows_tok) * unsigned(a.S), a.Hkv, a.B);
  LAZY_CUDA_TRY(launch_pdl(kern, grid, dim3(tc::kThreads), L::SMEM, st, mk, mv, a));
  return LAZY_OK;
}

template <bool SPLIT_V, bool KH>
static int dispatch_tc(int D, int kind, const CUtensorMap& mk, const CUtensorMap& mv, const tc::Args& a, int max_q,
                       cudaStream_t st) {
  if (D == 128) {
    if (kind == kRope) return launch_tc<128, kRope, SPLIT_V, KH>(mk, mv, a, max_q, st);
    if (kind == kRopeX) return launch_tc<128, kRopeX, SPLIT_V, KH>(mk, mv, a, max_q, st);
    if (kind == kAlibi) return launch_tc<128, kAlibi, SPLIT_V, KH>(mk, mv, a, max_q, st);
    return launch_tc<128, kNone, SPLIT_V, KH>(mk, mv, a, max_q, st);
  }
  if (kind == kRope) return launch_tc<64, kRope, SPLIT_V, KH>(mk, mv, a, max_q, st);
  if (kind == kRopeX) return launch_tc<64, kRopeX, SPLIT_V, KH>(mk, mv, a, max_q, st);
  if (kind == kAlibi) return launch_tc<64, kAlibi, SPLIT_V, KH>(mk, mv, a, max_q, st);
  return launch_tc<64, kNone, SPLIT_V, KH>(mk, mv, a, max_q, st);
}

int run_prefill_tc(const void* q, const int32_t* cu_q, const int32_t* q_start, const int32_t* doc_blocks,
                   const uint64_t* meta, int B, int max_blocks, int max_q, const void* k_cache,
                   const void* v_cache, int num_pages, int Hq, int Hkv, int D, const PosParams& pos, void* out,
                   float* lse, cudaStream_t st, const int32_t* seq_len, int S, float* part_o, float* part_ml) {
  const int G = Hq / Hkv;
  if (S < 1 || (S > 1 && (!seq_len || !part_o || !part_ml))) return fail(LAZY_EINVAL, "bad key-range split");
  if (G > tc::kM || (tc::kM % G) != 0) return fail(LAZY_EINVAL, "Hq/Hkv = %d must divide 128", G);
  CUtensorMap mk, mv;
  int rc = cache_map(&mk, k_cache, num_pages, Hkv, D);
  if (rc) return rc;
  rc = cache_map(&mv, v_cache, num_pages, Hkv, D);
  if (rc) return rc;
  tc::Args a;
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.cu_q = cu_q;
  a.q_start = q_start;
  a.doc_blocks = doc_blocks;
  a.meta = meta;
  a.B = B;
  a.max_blocks = max_blocks;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.num_pages = num_pages;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.lse = lse;
  a.status = status_word();
  a.pos = pos;
  a.seq_len = seq_len;
  a.S = S;
  a.part_o = part_o;
  a.part_ml = part_ml;
  if (seq_len) max_q = 1;
  // YaRN differs from RoPE only in its frequencies (already in pos.turns); partial rotary_dim or
  // interleaved pairs take the generic rotation (kRopeX)
  int kind = (pos.kind == kYarn) ? kRope : pos.kind;
  if (kind == kRope && (pos.rotary_dim != D || pos.interleaved)) kind = kRopeX;
  // A separate V producer when every CTA has one live Q tile (its tokens fit one 128-row tile)
  // and a long key range: at least 20 tiles of 128 keys per CTA.  Measured on GB300 (same-box
  // A/B): MQA decode 53.2 -> 49.6 us, yarn8b prefill 340 -> 323-330 us; rag8b's 16-tile CTAs
  // were slower with it.
  const int tiles_per_cta = ((max_blocks + tc::kPagesPerTile - 1) / tc::kPagesPerTile + S - 1) / S;
  const bool one_tile = seq_len != nullptr || max_q <= tc::kM / G;  // one live Q tile in every CTA
  const bool split_v = one_tile && tiles_per_cta >= 20;
  // With one live Q tile the second softmax warpgroup takes half of every tile's keys (KH).
  if (split_v) return dispatch_tc<true, true>(D, kind, mk, mv, a, max_q, st);
  if (one_tile) return dispatch_tc<false, true>(D, kind, mk, mv, a, max_q, st);
  return dispatch_tc<false, false>(D, kind, mk, mv, a, max_q, st);
}

}  // namespace lazykv
