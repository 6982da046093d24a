// Arguments of the split-KV decode kernel (also used for the per-row prefill path).
#pragma once

#include "common.cuh"

namespace lazykv {

struct DecodeArgs {
  const __nv_bfloat16* q;
  const int32_t* seq_len;
  const int32_t* cu_q;
  const int32_t* q_start;
  const int32_t* doc_blocks;
  const uint64_t* meta;
  const __nv_bfloat16* k_cache;
  const __nv_bfloat16* v_cache;
  int num_pages, B, max_blocks, Hq, Hkv, rows;
  int group;  // query heads per CTA (divides Hq / Hkv)
  int nw;     // warps per CTA (4, or 12 for small batches)
  __nv_bfloat16* out;
  float* lse;
  float* part_o;   // [rows][Hq][S][D]
  float* part_ml;  // [rows][Hq][S][2]
  int S;
  uint32_t* status;
  PosParams pos;
};

int run_decode_rows(DecodeArgs& a, int D, bool rows_mode, void* ws, size_t ws_bytes, cudaStream_t st);
struct DecodeShape {
  int nw;  // warps per CTA
  int S;   // KV splits per (row, head group)
};
DecodeShape decode_shape(int rows, int Hq, int Hkv, int max_blocks);
int choose_splits_rows(int rows, int Hq, int Hkv, int max_blocks);
// Workspace bytes of a decode (rows_mode = false) or of the CUDA-core prefill row mode.
size_t decode_ws_bytes(int rows, int Hq, int Hkv, int D, int max_blocks, bool rows_mode = false);
int run_prefill_tc(const void* q, const int32_t* cu_q, const int32_t* q_start, const int32_t* doc_blocks,
                   const uint64_t* meta, int B, int max_blocks, int max_q, const void* k_cache,
                   const void* v_cache, int num_pages, int Hq, int Hkv, int D, const PosParams& pos, void* out,
                   float* lse, cudaStream_t st, const int32_t* seq_len = nullptr, int S = 1,
                   float* part_o = nullptr, float* part_ml = nullptr);
// decode of wide head groups (Hq/Hkv >= 16) runs on the tensor-core kernel in decode mode
bool use_tc_decode(int Hq, int Hkv, int D);
int tc_decode_splits(int B, int Hkv, int max_blocks);

}  // namespace lazykv
