// Split-KV paged decode with deferred rotation (CUDA cores, HBM-bound).
//
// [NOTE] Tiling 感知的 Q/K 旋转分派: decode has M = 1, so rotating K would touch a whole tile;
// instead Q is rotated, and only when the KV block crosses a document boundary (the offset
// Delta changes).  [NOTE] 融合 Triton kernel + bit-packed 元数据: each block's (page, Delta,
// valid rows) is unpacked from one 64-bit word held in a register.  [GIST] Decoding: memory
// traffic stays that of plain paged attention (K and V only).
//
// Design (GB300):
//  * One CTA = (query row, head group, KV split); 4 warps (3 CTAs per SM), or 12 warps (one CTA
//    per SM, no split) when a small batch's units fill between half and all of the SMs.  Each
//    warp streams a contiguous run of pages through its own 2-stage ring of shared-memory
//    stages filled by cp.async.bulk (one 4 KB K copy and one V copy per page and head,
//    completed on an mbarrier).
//    No registers are spent on loads in flight, and every stage is in flight while earlier
//    pages are used.
//  * A lane owns 8 columns (one 16-byte chunk) of a K/V row; D/8 lanes cover a row.  Per page
//    every lane forms G x (rows per lane) partial dot products with packed fp32x2 FMAs, then a
//    transposed butterfly over the row's lanes leaves each lane with complete scores.
//  * q_eff = R_{m - Delta} q_raw, pre-multiplied by scale * log2(e), is recomputed in registers
//    when Delta changes (cos/sin from the table, or from exact fixed-point turns followed by the
//    SFU's sine/cosine).
//  * Online softmax in base 2 with a lazy max: the running max moves only when a score beats
//    it by more than 8 (a warp vote), so the common page needs no max reduction.
//  * Each CTA merges its warps; splits are merged by lse in a second small kernel, launched
//    with programmatic dependent launch so its launch overlaps this kernel's tail.
//  * "Rows" mode runs the same kernel with one query row per prefill token (causal limit
//    m = q_start + i): the simple correct prefill used for shapes without a tensor-core path.
#include <cfloat>

#include "decode.cuh"

namespace lazykv {

constexpr float kTau = 8.0f;  // lazy-rescale threshold (base-2 units)



// Transposed butterfly over the LPR lanes of a row group.  On return lane c (= lane % LPR)
// holds in v[0..E) the complete sums of indices c*E .. c*E+E-1 when V >= LPR, or of index
// c >> log2(LPR/V) (replicated over LPR/V lanes) when V < LPR.
template <int O, int CNT, int V>
struct RowReduce {
  static __device__ __forceinline__ void run(float (&v)[V], int lane) {
    if constexpr (O >= 1) {
      if constexpr (CNT > 1) {
        const bool up = (lane & O) != 0;
        constexpr int H = CNT / 2;
#pragma unroll
        for (int i = 0; i < H; ++i) {
          const float send = up ? v[i] : v[i + H];
          const float keep = up ? v[i + H] : v[i];
          v[i] = keep + __shfl_xor_sync(0xffffffffu, send, O);
        }
        RowReduce<O / 2, H, V>::run(v, lane);
      } else {
        v[0] += __shfl_xor_sync(0xffffffffu, v[0], O);
        RowReduce<O / 2, 1, V>::run(v, lane);
      }
    }
  }
};

template <int D, int G, int NST, int NW>  // NW warps per CTA
struct DecLayout {
  static constexpr int LPR = D / 8;             // lanes per row
  static constexpr int RPI = 32 / LPR;          // rows per warp-wide load
  static constexpr int RPL = kPage / RPI;       // rows per lane per page
  static constexpr int V = G * RPL;             // partial scores per lane per page
  static constexpr int E = V >= LPR ? V / LPR : 1;
  static constexpr int DUP = V >= LPR ? 1 : LPR / V;  // lanes holding the same score
  static constexpr int PAGE_BYTES = kPage * D * 2;
  static constexpr int STAGE_BYTES = 2 * PAGE_BYTES;
  static constexpr int STAGES_BYTES = NW * NST * STAGE_BYTES;
  static constexpr int QS_OFF = STAGES_BYTES;                 // q_raw fp32 [G][D]
  static constexpr int PB_OFF = QS_OFF + G * D * 4;           // p buffer [warp][16][G]
  static constexpr int SLOT_OFF = PB_OFF + NW * kPage * G * 4;  // [warp][NST] {u64 word, i32 rows}
  static constexpr int BAR_OFF = SLOT_OFF + NW * NST * 16;
  static constexpr int SMEM = BAR_OFF + NW * NST * 8;
  // after the page loop the stage area is reused to merge warps: [warp][G][D] o, [warp][G][2] m,l
  static_assert(NW * G * (D + 2) * 4 <= STAGES_BYTES, "merge buffer must fit in the stages");
  static_assert(SMEM <= 227 * 1024, "shared memory budget");
};

// NW = 4: the general shape, several CTAs per SM (3 for head groups of at most 4).
// NW = 12: one CTA per SM for launches whose (row, head group) units fit on the SMs (small
// batches): each unit gets a whole SM, so no SM holds more work than another.
template <int D, int G, int POS, bool ROWS, int NST, int NW>
__global__ void __launch_bounds__(NW * 32, (NW == 4 && G <= 4) ? 3 : 1) decode_kernel(const DecodeArgs a) {
  using L = DecLayout<D, G, NST, NW>;
  constexpr int LPR = L::LPR, RPI = L::RPI, RPL = L::RPL, V = L::V, E = L::E;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.x, hg = blockIdx.y, r = blockIdx.z;
  const int h0 = hg * G;                       // first query head of this CTA
  const int kvh = h0 / (a.Hq / a.Hkv);         // its KV head (contiguous GQA grouping)
  pdl_wait();

  // ---- the query row: request, absolute position m, visible blocks
  int b, m;
  const __nv_bfloat16* qrow;
  if constexpr (ROWS) {
    int lo = 0, hi = a.B;  // last b with cu_q[b] <= r
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (a.cu_q[mid] <= r) lo = mid; else hi = mid;
    }
    b = lo;
    m = a.q_start[b] + (r - a.cu_q[b]);
    qrow = a.q + (size_t)r * a.Hq * D;
  } else {
    b = r;
    m = a.seq_len[b] - 1;
    qrow = a.q + (size_t)b * a.Hq * D;
  }
  int nb = a.doc_blocks[b] + (m - a.q_start[b]) / kPage + 1;
  if (nb > a.max_blocks) {
    if (threadIdx.x == 0) set_status(a.status, LAZY_STATUS_BAD_ROW);
    nb = a.max_blocks;
  }
  const int chunk = (nb + a.S - 1) / a.S;
  const int beg = split * chunk, end = min(nb, beg + chunk);
  const int len = max(0, end - beg);
  // the warps' runs differ by at most one page
  const int wb = beg + warp * len / NW;
  const int n = beg + (warp + 1) * len / NW - wb;

  float* qs = reinterpret_cast<float*>(smem + L::QS_OFF);
  float* pbuf = reinterpret_cast<float*>(smem + L::PB_OFF) + warp * kPage * G;
  uint8_t* slots = smem + L::SLOT_OFF + warp * NST * 16;
  const uint32_t bar0 = smem_u32(smem + L::BAR_OFF + warp * NST * 8);
  const uint32_t stage0 = smem_u32(smem + warp * NST * L::STAGE_BYTES);

  // ---- block words of this warp's run, 32 at a time (coalesced), next chunk prefetched, and the
  // query values loaded into registers, so that the two latencies overlap; the first pages are
  // issued as soon as the block words arrive, before the query is staged in shared memory
  const uint64_t* mrow = a.meta + (size_t)b * a.max_blocks + wb;
  uint64_t mcur = lane < n ? ldg_u64(mrow + lane) : 0;
  uint64_t mnxt = 32 + lane < n ? ldg_u64(mrow + 32 + lane) : 0;
  int mbase = 0;
  constexpr int QPT = (G * D + NW * 32 - 1) / (NW * 32);  // query values per thread
  __nv_bfloat16 qv[QPT];
#pragma unroll
  for (int k = 0; k < QPT; ++k) {
    const int i = threadIdx.x + k * NW * 32;
    qv[k] = i < G * D ? qrow[h0 * D + i] : __float2bfloat16_rn(0.f);
  }
  if (lane == 0)
    for (int s = 0; s < NST; ++s) mbar_init(bar0 + 8 * s, 1);
  fence_mbar_init();
  __syncwarp();

  const size_t head_stride = (size_t)kPage * D;  // elements per (page, head)
  auto issue = [&](int i) {
    if (i >= mbase + 32) {
      mcur = mnxt;
      mbase += 32;
      mnxt = mbase + 32 + lane < n ? ldg_u64(mrow + mbase + 32 + lane) : 0;
    }
    const uint64_t w = __shfl_sync(0xffffffffu, mcur, i - mbase);
    const int st = i % NST;
    if (lane == 0) {
      const uint32_t page = word_page(w);
      const int start = int(word_delta(w) + kPage * word_pg(w));
      int rows = min(int(word_nvalid(w)), m - start + 1);
      rows = max(0, min(rows, kPage));
      if (page >= uint32_t(a.num_pages)) {
        set_status(a.status, LAZY_STATUS_BAD_PAGE);
        rows = 0;
      }
      *reinterpret_cast<uint64_t*>(slots + st * 16) = w;
      *reinterpret_cast<int*>(slots + st * 16 + 8) = rows;
      const uint32_t bytes = uint32_t(rows) * D * 2;
      const uint32_t bar = bar0 + 8 * st;
      mbar_arrive_expect_tx(bar, 2 * bytes);
      if (bytes) {
        const size_t off = ((size_t)page * a.Hkv + kvh) * head_stride;
        const uint32_t dst = stage0 + st * L::STAGE_BYTES;
        bulk_g2s(dst, a.k_cache + off, bytes, bar);
        bulk_g2s(dst + L::PAGE_BYTES, a.v_cache + off, bytes, bar);
      }
    }
  };

  const int pre = min(NST, n);
  for (int i = 0; i < pre; ++i) issue(i);
#pragma unroll
  for (int k = 0; k < QPT; ++k) {
    const int i = threadIdx.x + k * NW * 32;
    if (i < G * D) qs[i] = __bfloat162float(qv[k]);
  }
  __syncthreads();  // qs complete

  // ---- per-lane state
  const int c = lane % LPR;        // chunk (8 columns) of this lane
  const int c0 = c * 8;
  const int rg = lane / LPR;       // row group
  constexpr int kShift = (V >= LPR) ? 0 : (LPR / V == 2 ? 1 : LPR / V == 4 ? 2 : LPR / V == 8 ? 3 : 4);
  const int base_idx = (V >= LPR) ? c * E : (c >> kShift);
  const int h_lane = base_idx / RPL;  // the head of this lane's scores (E divides RPL)
  const bool unique = (V >= LPR) || ((c & (L::DUP - 1)) == 0);

  float2 qe[G][4];
  float2 o[G][4];
  float m_run[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    m_run[h] = -FLT_MAX;
#pragma unroll
    for (int e = 0; e < 4; ++e) o[h][e] = make_float2(0.f, 0.f);
  }
  float l_lane = 0.f;
  float alibi_lane = 0.f;
  if constexpr (POS == kAlibi) alibi_lane = a.pos.slopes[h0 + h_lane] * 1.4426950408889634f;
  if constexpr (POS == kAlibi || POS == kNone) {
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int e = 0; e < 4; ++e)
        qe[h][e] = make_float2(qs[h * D + c0 + 2 * e] * a.pos.scale_log2,
                               qs[h * D + c0 + 2 * e + 1] * a.pos.scale_log2);
  }
  uint32_t cur_delta = 0xFFFFFFFFu;
  bool first = true;

  for (int i = 0; i < n; ++i) {
    const int st = i % NST;
    const uint32_t bar = bar0 + 8 * st;
    if (!mbar_wait(bar, uint32_t((i / NST) & 1))) {
      if (lane == 0) set_status(a.status, LAZY_STATUS_TIMEOUT);
      for (int j = i + 1; j < min(n, i + NST); ++j) mbar_wait(bar0 + 8 * (j % NST), uint32_t((j / NST) & 1));
      break;
    }
    const uint64_t w = *reinterpret_cast<const uint64_t*>(slots + st * 16);
    const int rows_ok = *reinterpret_cast<const int*>(slots + st * 16 + 8);
    const uint32_t delta = word_delta(w);
    const int start = int(delta + kPage * word_pg(w));

    if constexpr (POS == kRope || POS == kYarn || POS == kRopeX) {
      if (delta != cur_delta) {  // document boundary: q_eff = R_{m - Delta} q_raw
        cur_delta = delta;
        const uint32_t dp = uint32_t(m) - delta;
        if constexpr (POS == kRopeX) {
          // Partial rotary_dim or interleaved pairs.  This lane's 8 columns c0..c0+7 are all of
          // one kind (rotary_dim is a multiple of 16): the first or second element of
          // half-split pairs (partner +-rd/2), adjacent interleaved pairs, or the unrotated tail.
          const int rd = a.pos.rotary_dim, hr = rd / 2;
          const bool inter = a.pos.interleaved != 0;
          const int kind = c0 >= rd ? 3 : inter ? 2 : (c0 < hr ? 0 : 1);
          const int f0 = kind == 2 ? c0 / 2 : (kind == 0 ? c0 : c0 - hr);  // first frequency
          const bool tab = a.pos.table != nullptr && int(dp) < a.pos.max_pos;
          float cs[8], sn[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int fi = f0 + (kind == 2 ? e / 2 : e);
            if (kind == 3) {
              cs[e] = 1.f;
              sn[e] = 0.f;
            } else if (tab) {
              cs[e] = a.pos.table[(size_t)dp * rd + fi];
              sn[e] = a.pos.table[(size_t)dp * rd + hr + fi];
            } else {
              turn_sincos_fast(dp, a.pos.turns[fi], sn[e], cs[e]);
            }
          }
#pragma unroll
          for (int h = 0; h < G; ++h) {
            const float* qh = qs + h * D;
            float y[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float x = qh[c0 + e];
              float v;
              if (kind == 0) v = x * cs[e] - qh[c0 + e + hr] * sn[e];
              else if (kind == 1) v = qh[c0 + e - hr] * sn[e] + x * cs[e];
              else if (kind == 2) v = (e & 1) ? qh[c0 + e - 1] * sn[e] + x * cs[e] : x * cs[e] - qh[c0 + e + 1] * sn[e];
              else v = x;
              y[e] = v * a.pos.scale_log2;
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) qe[h][e] = make_float2(y[2 * e], y[2 * e + 1]);
          }
        } else {
          // full-width half-split pairs (i, i + D/2)
          const bool first_half = c0 < D / 2;
          const int i0 = first_half ? c0 : c0 - D / 2;
          const bool tab = a.pos.table != nullptr && int(dp) < a.pos.max_pos;
          float cs[8], sn[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            if (tab) {
              cs[e] = a.pos.table[(size_t)dp * D + i0 + e];
              sn[e] = a.pos.table[(size_t)dp * D + D / 2 + i0 + e];
            } else {
              turn_sincos_fast(dp, a.pos.turns[i0 + e], sn[e], cs[e]);
            }
          }
#pragma unroll
          for (int h = 0; h < G; ++h) {
            float y[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float x1 = qs[h * D + i0 + e], x2 = qs[h * D + i0 + e + D / 2];
              y[e] = (first_half ? (x1 * cs[e] - x2 * sn[e]) : (x1 * sn[e] + x2 * cs[e])) * a.pos.scale_log2;
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) qe[h][e] = make_float2(y[2 * e], y[2 * e + 1]);
          }
        }
      }
    }

    // ---- scores: partial dots over this lane's 8 columns, head-major index h*RPL + rr
    const uint8_t* kp = smem + warp * NST * L::STAGE_BYTES + st * L::STAGE_BYTES;
    const uint8_t* vp = kp + L::PAGE_BYTES;
    float part[V];
#pragma unroll
    for (int rr = 0; rr < RPL; ++rr) {
      const int row = rr * RPI + rg;
      const uint4 kv = *reinterpret_cast<const uint4*>(kp + row * D * 2 + c0 * 2);
      const float2 k0 = bf2_to_f2(kv.x), k1 = bf2_to_f2(kv.y), k2 = bf2_to_f2(kv.z), k3 = bf2_to_f2(kv.w);
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float2 acc = __fmul2_rn(k0, qe[h][0]);
        acc = __ffma2_rn(k1, qe[h][1], acc);
        acc = __ffma2_rn(k2, qe[h][2], acc);
        acc = __ffma2_rn(k3, qe[h][3], acc);
        part[h * RPL + rr] = acc.x + acc.y;
      }
    }
    RowReduce<LPR / 2, V, V>::run(part, lane);

    // ---- this lane's complete scores: head h_lane, rows (base_idx + e) % RPL
    float s2[E];
    bool need = false;
    float mr = m_run[0];
#pragma unroll
    for (int h = 1; h < G; ++h)
      if (h == h_lane) mr = m_run[h];
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int rr = (base_idx + e) % RPL;
      const int row = rr * RPI + rg;
      float s = part[e];
      if constexpr (POS == kAlibi) s += alibi_lane * float(start + row - m);
      s2[e] = row < rows_ok ? s : -INFINITY;
      need |= s2[e] > mr + kTau;
    }
    if (__any_sync(0xffffffffu, need || first)) {
      first = false;
      float lm = -INFINITY;
#pragma unroll
      for (int e = 0; e < E; ++e) lm = fmaxf(lm, s2[e]);
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float x = (h == h_lane) ? lm : -INFINITY;
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, off));
        if (x > m_run[h]) {
          const float alpha = exp2f(m_run[h] - x);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            o[h][e].x *= alpha;
            o[h][e].y *= alpha;
          }
          if (h == h_lane) l_lane *= alpha;
          m_run[h] = x;
        }
      }
#pragma unroll
      for (int h = 1; h < G; ++h)
        if (h == h_lane) mr = m_run[h];
      if (h_lane == 0) mr = m_run[0];
    }
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int rr = (base_idx + e) % RPL;
      const int row = rr * RPI + rg;
      const float p = ex2_approx(s2[e] - mr);
      if (unique) {
        l_lane += p;
        pbuf[row * G + h_lane] = p;
      }
    }
    __syncwarp();

    // ---- O += P V over this lane's 8 columns, every head
#pragma unroll
    for (int rr = 0; rr < RPL; ++rr) {
      const int row = rr * RPI + rg;
      if (row < rows_ok) {
        const uint4 vv = *reinterpret_cast<const uint4*>(vp + row * D * 2 + c0 * 2);
        const float2 v0 = bf2_to_f2(vv.x), v1 = bf2_to_f2(vv.y), v2 = bf2_to_f2(vv.z), v3 = bf2_to_f2(vv.w);
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float p = pbuf[row * G + h];
          const float2 pp = make_float2(p, p);
          o[h][0] = __ffma2_rn(v0, pp, o[h][0]);
          o[h][1] = __ffma2_rn(v1, pp, o[h][1]);
          o[h][2] = __ffma2_rn(v2, pp, o[h][2]);
          o[h][3] = __ffma2_rn(v3, pp, o[h][3]);
        }
      }
    }
    __syncwarp();
    if (i + NST < n) issue(i + NST);
  }

  pdl_trigger();  // every CTA of the grid is running once all have reached this point

  // ---- fold row groups, then the warps of the CTA
#pragma unroll
  for (int off = LPR; off < 32; off <<= 1)
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        o[h][e].x += __shfl_xor_sync(0xffffffffu, o[h][e].x, off);
        o[h][e].y += __shfl_xor_sync(0xffffffffu, o[h][e].y, off);
      }
  float l_head[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    float x = (h == h_lane && unique) ? l_lane : 0.f;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    l_head[h] = x;
  }
  __syncthreads();  // every stage consumed: reuse the stage area
  float* mo = reinterpret_cast<float*>(smem);                  // [warp][G][D]
  float* mml = mo + NW * G * D;                                  // [warp][G][2]
  if (lane < LPR) {
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        mo[(warp * G + h) * D + c0 + 2 * e] = o[h][e].x;
        mo[(warp * G + h) * D + c0 + 2 * e + 1] = o[h][e].y;
      }
  }
  if (lane == 0) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      mml[(warp * G + h) * 2] = (l_head[h] > 0.f) ? m_run[h] : -INFINITY;
      mml[(warp * G + h) * 2 + 1] = l_head[h];
    }
  }
  __syncthreads();
  for (int t = threadIdx.x; t < G * D; t += blockDim.x) {
    const int h = t / D, col = t % D;
    float M = -INFINITY;
#pragma unroll
    for (int w2 = 0; w2 < NW; ++w2) M = fmaxf(M, mml[(w2 * G + h) * 2]);
    float Ov = 0.f, Lv = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w2 = 0; w2 < NW; ++w2) {
        const float mw = mml[(w2 * G + h) * 2];
        const float sc = mw == -INFINITY ? 0.f : exp2f(mw - M);
        Ov += sc * mo[(w2 * G + h) * D + col];
        Lv += sc * mml[(w2 * G + h) * 2 + 1];
      }
    }
    const int hq = h0 + h;
    if (a.S == 1) {
      const float inv = Lv > 0.f ? 1.f / Lv : 0.f;
      a.out[((size_t)r * a.Hq + hq) * D + col] = __float2bfloat16_rn(Ov * inv);
      if (a.lse && col == 0) a.lse[(size_t)r * a.Hq + hq] = (M + log2f(Lv)) * 0.6931471805599453f;
    } else {
      const size_t pi = ((size_t)r * a.Hq + hq) * a.S + split;
      a.part_o[pi * D + col] = Ov;
      if (col == 0) {
        a.part_ml[pi * 2] = M;
        a.part_ml[pi * 2 + 1] = Lv;
      }
    }
  }
}

// Merge S partial (O, m, l) per (row, head) by their log-sum-exp (flash-decoding style).
template <int D>
__global__ void __launch_bounds__(D) merge_kernel(const float* __restrict__ part_o, const float* __restrict__ part_ml,
                                                  int S, int Hq, __nv_bfloat16* __restrict__ out,
                                                  float* __restrict__ lse) {
  pdl_wait();
  pdl_trigger();
  const size_t rh = blockIdx.x;  // row * Hq + head
  const int col = threadIdx.x;
  const float* ml = part_ml + rh * S * 2;
  float M = -INFINITY;
  for (int s = 0; s < S; ++s) M = fmaxf(M, ml[2 * s]);
  float Ov = 0.f, Lv = 0.f;
  if (M != -INFINITY) {
    for (int s = 0; s < S; ++s) {
      const float ms = ml[2 * s];
      const float sc = ms == -INFINITY ? 0.f : exp2f(ms - M);
      Ov += sc * part_o[(rh * S + s) * D + col];
      Lv += sc * ml[2 * s + 1];
    }
  }
  out[rh * D + col] = __float2bfloat16_rn(Lv > 0.f ? Ov / Lv : 0.f);
  if (lse && col == 0) lse[rh] = (M + log2f(Lv)) * 0.6931471805599453f;
}

// ------------------------------------------------------------------------------------------
// Host: split choice, workspace, dispatch
// ------------------------------------------------------------------------------------------
// Two stages per warp: 4 warps x 2 x 8 KB keeps a CTA at ~68 KB of shared memory and <= 168
// registers (G <= 4), so three CTAs fit per SM; measured on GB300 against three stages at two
// CTAs per SM: decode32k 1324 -> 1223 us, yarn8b 294 -> 267 us, rag8b unchanged.
constexpr int kNst = 2;

int decode_group(int Hq, int Hkv) {
  const int G = Hq / Hkv;
  return G >= 8 ? 8 : G;  // heads per CTA (MQA: several CTAs share one KV head)
}

// Warps per CTA and KV splits of the CUDA-core decode.
DecodeShape decode_shape(int rows, int Hq, int Hkv, int max_blocks) {
  const int G = decode_group(Hq, Hkv);
  const long long units = (long long)rows * (Hq / G);
  const int sms = sm_count();
  // Small batches whose (row, head group) units fill between half and all of the SMs: one
  // 12-warp CTA per unit, no key split.  Every SM then carries the same load (three 4-warp CTAs
  // on some SMs and two on others did not), and there is no partial to merge.  Fewer units are
  // better served by 4-warp CTAs split over more SMs.
  if (G <= 4 && units <= sms && 2 * units > sms && max_blocks >= 12 * 4) return {12, 1};
  return {4, choose_splits_rows(rows, Hq, Hkv, max_blocks)};
}

// Splits of the 4-warp shape (also the CUDA-core prefill's row mode, one query row per unit).
int choose_splits_rows(int rows, int Hq, int Hkv, int max_blocks) {
  const int G = decode_group(Hq, Hkv);
  const long long units = (long long)rows * (Hq / G);
  const long long slots = (long long)sm_count() * (G <= 4 ? 3 : 2);  // 4-warp CTAs resident at once
  // About 4 waves of resident CTAs, but runs of about 16 pages per warp: measured on GB300,
  // long per-warp page runs beat more, shorter CTAs (every CTA pays a pipeline start-up and its
  // split partials), and a partial last wave costs little once there are several waves.
  const long long want = (4 * slots + units - 1) / units;
  const int max_by_len = max(1, (max_blocks + 4 * 16 - 1) / (4 * 16));
  long long s = want < max_by_len ? want : max_by_len;
  if (s < 1) s = 1;
  if (s > 64) s = 64;
  return int(s);
}

// Wide head groups (MQA-like, G >= 16): per page the CUDA-core kernel would spread the group
// over G/8 CTAs that each re-read K/V and spend G x 4 KB of FMAs per page, so these rows go
// to the tensor-core kernel instead, with the G heads of the new token as its query rows.
bool use_tc_decode(int Hq, int Hkv, int D) {
  const int G = Hq / Hkv;
  return G >= 16 && 128 % G == 0 && (D == 64 || D == 128);
}

// Key-range splits of the tensor-core decode: one wave of single-CTA-per-SM units, at least
// four 128-key tiles per split.
int tc_decode_splits(int B, int Hkv, int max_blocks) {
  const long long units = (long long)B * Hkv;
  const int tiles = (max_blocks + 7) / 8;
  long long s = sm_count() / (units > 0 ? units : 1);
  if (s > tiles / 4) s = tiles / 4;
  if (s < 1) s = 1;
  if (s > 64) s = 64;
  return int(s);
}

size_t decode_ws_bytes(int rows, int Hq, int Hkv, int D, int max_blocks, bool rows_mode) {
  const int S = rows_mode                    ? choose_splits_rows(rows, Hq, Hkv, max_blocks)
                : use_tc_decode(Hq, Hkv, D) ? tc_decode_splits(rows, Hkv, max_blocks)
                                            : decode_shape(rows, Hq, Hkv, max_blocks).S;
  if (S <= 1) return 0;
  const size_t po = (size_t)rows * Hq * S * D * 4;
  const size_t pml = (size_t)rows * Hq * S * 2 * 4;
  return ((po + 255) / 256) * 256 + pml;
}

template <int D, int G, int POS, bool ROWS, int NW>
static int launch_nw(const DecodeArgs& a, cudaStream_t st) {
  using L = DecLayout<D, G, kNst, NW>;
  auto kern = decode_kernel<D, G, POS, ROWS, kNst, NW>;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (!attr_set[dev & 63]) {
    LAZY_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM));
    attr_set[dev & 63] = true;
  }
  dim3 grid(a.S, a.Hq / G, a.rows);
  LAZY_CUDA_TRY(launch_pdl(kern, grid, dim3(NW * 32), L::SMEM, st, a));
  if (a.S > 1)
    LAZY_CUDA_TRY(launch_pdl(merge_kernel<D>, dim3((unsigned)a.rows * a.Hq), dim3(D), 0, st,
                             (const float*)a.part_o, (const float*)a.part_ml, a.S, a.Hq, a.out, a.lse));
  return LAZY_OK;
}

template <int D, int G, int POS, bool ROWS>
static int launch_t(const DecodeArgs& a, cudaStream_t st) {
  if constexpr (G <= 4 && !ROWS)
    if (a.nw == 12) return launch_nw<D, G, POS, ROWS, 12>(a, st);
  return launch_nw<D, G, POS, ROWS, 4>(a, st);
}

template <int D, int G, bool ROWS>
static int launch_pos(const DecodeArgs& a, cudaStream_t st) {
  switch (a.pos.kind) {
    case kRope:
    case kYarn:
      if (a.pos.rotary_dim != D || a.pos.interleaved) return launch_t<D, G, kRopeX, ROWS>(a, st);
      return launch_t<D, G, kRope, ROWS>(a, st);
    case kAlibi: return launch_t<D, G, kAlibi, ROWS>(a, st);
    default: return launch_t<D, G, kNone, ROWS>(a, st);
  }
}

template <int D, bool ROWS>
static int launch_g(const DecodeArgs& a, cudaStream_t st) {
  switch (a.group) {
    case 1: return launch_pos<D, 1, ROWS>(a, st);
    case 2: return launch_pos<D, 2, ROWS>(a, st);
    case 4: return launch_pos<D, 4, ROWS>(a, st);
    case 8: return launch_pos<D, 8, ROWS>(a, st);
    default: return fail(LAZY_EINVAL, "unsupported heads per CTA %d", a.group);
  }
}

int run_decode_rows(DecodeArgs& a, int D, bool rows_mode, void* ws, size_t ws_bytes, cudaStream_t st) {
  if (!rows_mode && use_tc_decode(a.Hq, a.Hkv, D)) {
    a.S = tc_decode_splits(a.rows, a.Hkv, a.max_blocks);
    if (a.S > 1) {
      const size_t need = decode_ws_bytes(a.rows, a.Hq, a.Hkv, D, a.max_blocks, false);
      if (!ws || ws_bytes < need)
        return fail(LAZY_EINVAL, "workspace too small: need %zu bytes, got %zu", need, ws_bytes);
      if (reinterpret_cast<uintptr_t>(ws) & 255u) return fail(LAZY_EINVAL, "workspace must be 256-byte aligned");
      const size_t po = (size_t)a.rows * a.Hq * a.S * D * 4;
      a.part_o = static_cast<float*>(ws);
      a.part_ml = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + ((po + 255) / 256) * 256);
    }
    int rc = run_prefill_tc(a.q, nullptr, a.q_start, a.doc_blocks, a.meta, a.B, a.max_blocks, 1, a.k_cache,
                            a.v_cache, a.num_pages, a.Hq, a.Hkv, D, a.pos, a.out, a.lse, st, a.seq_len, a.S,
                            a.part_o, a.part_ml);
    if (rc || a.S == 1) return rc;
    if (D == 128)
      LAZY_CUDA_TRY(launch_pdl(merge_kernel<128>, dim3((unsigned)a.rows * a.Hq), dim3(128), 0, st,
                               (const float*)a.part_o, (const float*)a.part_ml, a.S, a.Hq, a.out, a.lse));
    else
      LAZY_CUDA_TRY(launch_pdl(merge_kernel<64>, dim3((unsigned)a.rows * a.Hq), dim3(64), 0, st,
                               (const float*)a.part_o, (const float*)a.part_ml, a.S, a.Hq, a.out, a.lse));
    return LAZY_OK;
  }
  a.group = decode_group(a.Hq, a.Hkv);
  const int G = a.Hq / a.Hkv;
  if (G % a.group != 0) return fail(LAZY_EINVAL, "Hq/Hkv = %d not supported", G);
  const DecodeShape shp = rows_mode ? DecodeShape{4, choose_splits_rows(a.rows, a.Hq, a.Hkv, a.max_blocks)}
                                    : decode_shape(a.rows, a.Hq, a.Hkv, a.max_blocks);
  a.nw = shp.nw;
  a.S = shp.S;
  if (a.S > 1) {
    const size_t need = decode_ws_bytes(a.rows, a.Hq, a.Hkv, D, a.max_blocks, rows_mode);
    if (!ws || ws_bytes < need)
      return fail(LAZY_EINVAL, "workspace too small: need %zu bytes, got %zu", need, ws_bytes);
    if (reinterpret_cast<uintptr_t>(ws) & 255u) return fail(LAZY_EINVAL, "workspace must be 256-byte aligned");
    const size_t po = (size_t)a.rows * a.Hq * a.S * D * 4;
    a.part_o = static_cast<float*>(ws);
    a.part_ml = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + ((po + 255) / 256) * 256);
  }
  if (D == 128) return rows_mode ? launch_g<128, true>(a, st) : launch_g<128, false>(a, st);
  return rows_mode ? launch_g<64, true>(a, st) : launch_g<64, false>(a, st);
}

}  // namespace lazykv
