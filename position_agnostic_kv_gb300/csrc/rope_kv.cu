// cos/sin table and the position-free KV write.
//
// [NOTE] 整体框架: the cache holds each document indexed from its own local position 0, so a
// key is stored as R_j k with j its position inside the document; the attention kernels later
// apply one relative rotation R_Delta.  [NOTE] Tiling 感知: cos/sin come from a table (one
// D-length row per offset) or are computed on the fly.
#include "common.cuh"

namespace lazykv {

// Row p of the table: cos(p theta_i) for i < d/2, then sin(p theta_i).
__global__ void rope_table_kernel(PosParams pos, int max_pos, float* __restrict__ out) {
  const int half = pos.rotary_dim / 2;
  const long long n = (long long)max_pos * half;
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < n;
       idx += (long long)gridDim.x * blockDim.x) {
    const int p = int(idx / half), i = int(idx % half);
    float s, c;
    turn_sincos(uint32_t(p), pos.turns[i], s, c);
    out[(long long)p * pos.rotary_dim + i] = c;
    out[(long long)p * pos.rotary_dim + half + i] = s;
  }
}

// cos / sin of frequency i at position j (table row j: cos of the rotary_dim/2 frequencies,
// then their sin), or on the fly from exact turns.
__device__ __forceinline__ void pos_cs(const PosParams& pos, uint32_t j, bool use_table, int i, float& s, float& c) {
  if (use_table) {
    c = pos.table[(long long)j * pos.rotary_dim + i];
    s = pos.table[(long long)j * pos.rotary_dim + pos.rotary_dim / 2 + i];
  } else {
    turn_sincos(j, pos.turns[i], s, c);
  }
}

// One thread per (token, head, pair of 16-byte chunks); D/16 threads per (t, h).  Half-split
// RoPE: thread `part` < rotary_dim/16 rotates chunk `part` against its partner
// `part + rotary_dim/16` (pairs (i, i + rotary_dim/2)); the other threads copy the unrotated
// tail two chunks at a time.  Interleaved RoPE: thread `part` takes chunks 2 part and
// 2 part + 1 and rotates the adjacent pairs of those below rotary_dim.  fp32 math, one
// rounding to bf16; V is copied.
template <int D, bool ROTATE>
__global__ void __launch_bounds__(256) kv_write_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                                                       const int32_t* __restrict__ slot,
                                                       const int32_t* __restrict__ local_pos, int T,
                                                       int Hkv, uint4* __restrict__ kc, uint4* __restrict__ vc,
                                                       int num_pages, PosParams pos, uint32_t* status) {
  constexpr int TPR = D / 16;       // threads per (token, head)
  constexpr int CH = D / 8;         // 16-byte chunks per row
  pdl_wait();
  pdl_trigger();  // one small wave: every CTA is running
  const long long gid = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  const long long row = gid / TPR;  // (token, head)
  const int part = int(gid % TPR);
  if (row >= (long long)T * Hkv) return;
  const int t = int(row / Hkv), h = int(row % Hkv);
  const int sl = slot[t];
  if (sl < 0 || sl >= num_pages * kPage) {
    if (part == 0) set_status(status, LAZY_STATUS_BAD_SLOT);
    return;
  }
  const int page = sl / kPage, r = sl % kPage;
  const long long src = row * CH;
  const long long dst = (((long long)page * Hkv + h) * kPage + r) * CH;
  const int hc = pos.rotary_dim / 16;  // half-split: rotated chunk pairs
  const bool half_pair = ROTATE && !pos.interleaved && part < hc;
  int c1 = 2 * part, c2 = 2 * part + 1;
  if (ROTATE && !pos.interleaved) {
    c1 = half_pair ? part : 2 * hc + 2 * (part - hc);
    c2 = half_pair ? part + hc : c1 + 1;
  }
  uint4 a = k[src + c1], b = k[src + c2];
  if (ROTATE) {
    const uint32_t j = uint32_t(local_pos[t]);
    const bool use_table = pos.table != nullptr && int(j) < pos.max_pos;
    uint32_t* pa = reinterpret_cast<uint32_t*>(&a);
    uint32_t* pb = reinterpret_cast<uint32_t*>(&b);
    if (half_pair) {
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        float x1[2] = {bf_lo(pa[w]), bf_hi(pa[w])};
        float x2[2] = {bf_lo(pb[w]), bf_hi(pb[w])};
        float y1[2], y2[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float s, c;
          pos_cs(pos, j, use_table, part * 8 + w * 2 + e, s, c);  // pair index
          y1[e] = x1[e] * c - x2[e] * s;
          y2[e] = x1[e] * s + x2[e] * c;
        }
        pa[w] = f2_to_bf2(y1[0], y1[1]);
        pb[w] = f2_to_bf2(y2[0], y2[1]);
      }
    } else if (pos.interleaved) {
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int cc = q ? c2 : c1;
        uint32_t* pw = q ? pb : pa;
        if (cc < pos.rotary_dim / 8) {
#pragma unroll
          for (int w = 0; w < 4; ++w) {  // word w = (x_2i, x_2i+1), pair i = 4 cc + w
            float s, c;
            pos_cs(pos, j, use_table, cc * 4 + w, s, c);
            const float x0 = bf_lo(pw[w]), x1 = bf_hi(pw[w]);
            pw[w] = f2_to_bf2(x0 * c - x1 * s, x0 * s + x1 * c);
          }
        }
      }
    }
  }
  kc[dst + c1] = a;
  kc[dst + c2] = b;
  vc[dst + c1] = v[src + c1];
  vc[dst + c2] = v[src + c2];
}

}  // namespace lazykv

using namespace lazykv;

extern "C" int lazy_build_rope_table(const lazy_pos_cfg* cfg, int max_pos, float* out_table, void* stream) {
  int rc = check_device();
  if (rc) return rc;
  if (!cfg || !out_table || max_pos <= 0) return fail(LAZY_EINVAL, "bad rope table arguments");
  if (cfg->kind != LAZY_POS_ROPE && cfg->kind != LAZY_POS_YARN)
    return fail(LAZY_EINVAL, "a cos/sin table exists only for RoPE and YaRN");
  if (cfg->rotary_dim < 16 || cfg->rotary_dim > 128 || cfg->rotary_dim % 16)
    return fail(LAZY_EINVAL, "rotary_dim must be a multiple of 16 in [16, 128]");
  PosParams pos;
  lazy_pos_cfg c2 = *cfg;
  c2.cos_sin = nullptr;
  rc = prepare_pos(&c2, 1, cfg->rotary_dim, 0.f, &pos);
  if (rc) return rc;
  const long long n = (long long)max_pos * (cfg->rotary_dim / 2);
  const int threads = 256;
  const long long want = (n + threads - 1) / threads;
  const int blocks = int(want < 4L * 1024 * 152 ? want : 4L * 1024 * 152);
  rope_table_kernel<<<blocks, threads, 0, static_cast<cudaStream_t>(stream)>>>(pos, max_pos, out_table);
  LAZY_CUDA_TRY(cudaGetLastError());
  return LAZY_OK;
}

extern "C" int lazy_kv_write(const void* k, const void* v, const int32_t* slot, const int32_t* local_pos,
                             int T, int Hkv, int D, void* k_cache, void* v_cache, int num_pages,
                             const lazy_pos_cfg* cfg, void* stream) {
  int rc = check_device();
  if (rc) return rc;
  if (T < 0 || Hkv <= 0 || num_pages <= 0) return fail(LAZY_EINVAL, "bad kv_write sizes");
  if (D != 64 && D != 128) return fail(LAZY_EINVAL, "head_dim must be 64 or 128, got %d", D);
  if (T == 0) return LAZY_OK;
  if (!k || !v || !slot || !k_cache || !v_cache) return fail(LAZY_EINVAL, "NULL pointer");
  auto al = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  if (!al(k) || !al(v) || !al(k_cache) || !al(v_cache)) return fail(LAZY_EINVAL, "tensors must be 16-byte aligned");
  PosParams pos;
  rc = prepare_pos(cfg, 1, D, 0.f, &pos);
  if (rc) return rc;
  const bool rotate = pos.kind == kRope || pos.kind == kYarn;
  if (rotate && !local_pos) return fail(LAZY_EINVAL, "local_pos is NULL");
  const long long threads_total = (long long)T * Hkv * (D / 16);
  const int threads = 256;
  const int blocks = int((threads_total + threads - 1) / threads);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t* status = status_word();
  const uint4* k4 = static_cast<const uint4*>(k);
  const uint4* v4 = static_cast<const uint4*>(v);
  uint4* kc = static_cast<uint4*>(k_cache);
  uint4* vc = static_cast<uint4*>(v_cache);
  auto kern = D == 128 ? (rotate ? kv_write_kernel<128, true> : kv_write_kernel<128, false>)
                       : (rotate ? kv_write_kernel<64, true> : kv_write_kernel<64, false>);
  LAZY_CUDA_TRY(launch_pdl(kern, dim3(blocks), dim3(threads), 0, st, k4, v4, slot, local_pos, T, Hkv, kc, vc,
                           num_pages, pos, status));
  return LAZY_OK;
}
