// extern "C" entry points of the attention kernels: argument checks and dispatch.
#include "decode.cuh"

using namespace lazykv;

static int check_common(int B, int max_blocks, int Hq, int Hkv, int D, int num_pages, const void* kc,
                        const void* vc, const void* q, const void* out, const uint64_t* meta) {
  if (B < 0 || max_blocks <= 0 || Hq <= 0 || Hkv <= 0 || num_pages <= 0)
    return fail(LAZY_EINVAL, "bad sizes (B=%d max_blocks=%d Hq=%d Hkv=%d num_pages=%d)", B, max_blocks, Hq, Hkv,
                num_pages);
  if (D != 64 && D != 128) return fail(LAZY_EINVAL, "head_dim must be 64 or 128, got %d", D);
  if (Hq % Hkv) return fail(LAZY_EINVAL, "Hq (%d) must be a multiple of Hkv (%d)", Hq, Hkv);
  const int G = Hq / Hkv;
  if (G > 8 && G % 8) return fail(LAZY_EINVAL, "Hq/Hkv = %d: above 8 it must be a multiple of 8", G);
  if (G < 8 && (G & (G - 1))) return fail(LAZY_EINVAL, "Hq/Hkv = %d must be a power of two below 8", G);
  if (uint64_t(num_pages) > (1ull << 24)) return fail(LAZY_ERANGE, "num_pages above 2^24");
  auto al = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  if (!kc || !vc || !q || !out || !meta) return fail(LAZY_EINVAL, "NULL pointer");
  if (!al(kc) || !al(vc) || !al(q) || !al(out)) return fail(LAZY_EINVAL, "tensors must be 16-byte aligned");
  return LAZY_OK;
}

extern "C" int lazy_attn_decode(const void* q, const int32_t* seq_len, const int32_t* q_start,
                                const int32_t* doc_blocks, const uint64_t* meta, int B, int max_blocks,
                                const void* k_cache, const void* v_cache, int num_pages, int Hq, int Hkv,
                                int D, float scale, const lazy_pos_cfg* cfg, void* out, float* lse, void* ws,
                                size_t ws_bytes, void* stream) {
  int rc = check_device();
  if (rc) return rc;
  rc = check_common(B, max_blocks, Hq, Hkv, D, num_pages, k_cache, v_cache, q, out, meta);
  if (rc) return rc;
  if (B == 0) return LAZY_OK;
  if (!seq_len || !q_start || !doc_blocks) return fail(LAZY_EINVAL, "NULL metadata pointer");
  DecodeArgs a = {};
  rc = prepare_pos(cfg, Hq, D, scale, &a.pos);
  if (rc) return rc;
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.seq_len = seq_len;
  a.cu_q = nullptr;
  a.q_start = q_start;
  a.doc_blocks = doc_blocks;
  a.meta = meta;
  a.k_cache = static_cast<const __nv_bfloat16*>(k_cache);
  a.v_cache = static_cast<const __nv_bfloat16*>(v_cache);
  a.num_pages = num_pages;
  a.B = B;
  a.max_blocks = max_blocks;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.rows = B;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.lse = lse;
  a.status = status_word();
  return run_decode_rows(a, D, false, ws, ws_bytes, static_cast<cudaStream_t>(stream));
}

extern "C" int lazy_attn_prefill(const void* q, const int32_t* cu_q, const int32_t* q_start,
                                 const int32_t* doc_blocks, const uint64_t* meta, int B, int max_blocks,
                                 int total_q, int max_q, const void* k_cache, const void* v_cache, int num_pages,
                                 int Hq, int Hkv, int D, float scale, const lazy_pos_cfg* cfg, void* out,
                                 float* lse, void* ws, size_t ws_bytes, void* stream) {
  int rc = check_device();
  if (rc) return rc;
  rc = check_common(B, max_blocks, Hq, Hkv, D, num_pages, k_cache, v_cache, q, out, meta);
  if (rc) return rc;
  if (total_q < 0 || max_q < 0) return fail(LAZY_EINVAL, "bad total_q / max_q");
  if (B == 0 || total_q == 0) return LAZY_OK;
  if (!cu_q || !q_start || !doc_blocks) return fail(LAZY_EINVAL, "NULL metadata pointer");
  DecodeArgs a = {};
  rc = prepare_pos(cfg, Hq, D, scale, &a.pos);
  if (rc) return rc;
  const int G = Hq / Hkv;
  if (G <= 128 && 128 % G == 0)  // tensor-core path: 128 GQA-packed query rows per CTA
    return run_prefill_tc(q, cu_q, q_start, doc_blocks, meta, B, max_blocks, max_q, k_cache, v_cache, num_pages,
                          Hq, Hkv, D, a.pos, out, lse, static_cast<cudaStream_t>(stream));
  // other head groupings: one CTA per query row on CUDA cores (the decode kernel's row mode)
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.seq_len = nullptr;
  a.cu_q = cu_q;
  a.q_start = q_start;
  a.doc_blocks = doc_blocks;
  a.meta = meta;
  a.k_cache = static_cast<const __nv_bfloat16*>(k_cache);
  a.v_cache = static_cast<const __nv_bfloat16*>(v_cache);
  a.num_pages = num_pages;
  a.B = B;
  a.max_blocks = max_blocks;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.rows = total_q;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.lse = lse;
  a.status = status_word();
  return run_decode_rows(a, D, true, ws, ws_bytes, static_cast<cudaStream_t>(stream));
}

extern "C" size_t lazy_workspace_size(int phase, int rows, int B, int max_blocks, int Hq, int Hkv, int D) {
  (void)B;
  if (rows <= 0 || max_blocks <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv) return 0;
  if (phase == LAZY_PHASE_DECODE) return decode_ws_bytes(rows, Hq, Hkv, D, max_blocks);
  if (phase != LAZY_PHASE_PREFILL) return 0;
  const int G = Hq / Hkv;
  if (G <= 128 && 128 % G == 0) return 0;  // the tensor-core prefill needs no workspace
  return decode_ws_bytes(rows, Hq, Hkv, D, max_blocks, true);
}
