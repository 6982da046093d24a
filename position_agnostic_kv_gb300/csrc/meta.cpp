// lazy_build_doc_meta: the per-request block list with one packed 64-bit word per block.
//
// [README] Variants: the scheduler builds per-request rotation metadata.  [NOTE] 融合 Triton
// kernel + bit-packed 元数据: (block id, offset, mask) live in one 64-bit register and are
// unpacked with shifts.  [NOTE] 整体框架: every document is cached from local position 0 and a
// request places it at the offset Delta = total length of the documents before it.
//
// Word layout (LSB first): [4:0] n_valid, [15:5] pg (page index within the document),
// [39:16] Delta, [63:40] physical page.  Only a document's last page can be partial, so the
// "mask" of a block is the count n_valid of its leading valid rows.
#include <cstdint>
#include <cstring>

#include "lazykv.h"

namespace lazykv {
int fail(int code, const char* fmt, ...);
}

namespace {
constexpr int kPage = LAZY_PAGE_SIZE;
constexpr uint64_t kMaxPg = 1u << 11, kMaxDelta = 1u << 24, kMaxPage = 1u << 24;

inline uint64_t pack(uint32_t n_valid, uint32_t pg, uint32_t delta, uint32_t page) {
  return uint64_t(n_valid) | (uint64_t(pg) << 5) | (uint64_t(delta) << 16) | (uint64_t(page) << 40);
}
}  // namespace

extern "C" int lazy_build_doc_meta(int B, const int32_t* req_doc_off, const int32_t* req_docs,
                                   int n_docs, const int32_t* doc_len,
                                   const int32_t* doc_page_off, const int32_t* doc_pages,
                                   const int32_t* q_len, const int32_t* q_page_off,
                                   const int32_t* q_pages, int max_blocks, int32_t* block_table,
                                   uint64_t* meta, int32_t* seq_len, int32_t* q_start,
                                   int32_t* doc_blocks) {
  using lazykv::fail;
  if (B < 0 || max_blocks <= 0 || n_docs < 0) return fail(LAZY_EINVAL, "bad B / max_blocks / n_docs");
  if (B == 0) return LAZY_OK;
  if (!req_doc_off || !q_len || !q_page_off || !block_table || !meta || !seq_len || !q_start ||
      !doc_blocks)
    return fail(LAZY_EINVAL, "NULL argument");
  if (n_docs > 0 && (!doc_len || !doc_page_off)) return fail(LAZY_EINVAL, "NULL document arrays");
  std::memset(block_table, 0, sizeof(int32_t) * size_t(B) * size_t(max_blocks));
  std::memset(meta, 0, sizeof(uint64_t) * size_t(B) * size_t(max_blocks));
  for (int b = 0; b < B; ++b) {
    int32_t* bt = block_table + size_t(b) * max_blocks;
    uint64_t* mw = meta + size_t(b) * max_blocks;
    int j = 0;
    int64_t delta = 0;
    if (req_doc_off[b] > req_doc_off[b + 1]) return fail(LAZY_EINVAL, "req_doc_off not monotone at %d", b);
    for (int x = req_doc_off[b]; x < req_doc_off[b + 1]; ++x) {
      const int d = req_docs[x];
      if (d < 0 || d >= n_docs) return fail(LAZY_EINVAL, "request %d names document %d of %d", b, d, n_docs);
      const int L = doc_len[d];
      if (L < 0) return fail(LAZY_EINVAL, "document %d has negative length", d);
      const int npg = (L + kPage - 1) / kPage;
      if (doc_page_off[d + 1] - doc_page_off[d] < npg)
        return fail(LAZY_EINVAL, "document %d has %d pages, needs %d", d,
                    doc_page_off[d + 1] - doc_page_off[d], npg);
      if (uint64_t(npg) > kMaxPg) return fail(LAZY_ERANGE, "document %d longer than %d pages", d, int(kMaxPg));
      for (int pg = 0; pg < npg; ++pg) {
        if (j >= max_blocks) return fail(LAZY_ERANGE, "request %d needs more than max_blocks=%d", b, max_blocks);
        const int32_t page = doc_pages[doc_page_off[d] + pg];
        if (page < 0 || uint64_t(page) >= kMaxPage) return fail(LAZY_ERANGE, "page id %d out of range", page);
        if (uint64_t(delta) >= kMaxDelta) return fail(LAZY_ERANGE, "offset %lld >= 2^24", (long long)delta);
        const int n_valid = (L - kPage * pg) < kPage ? (L - kPage * pg) : kPage;
        mw[j] = pack(uint32_t(n_valid), uint32_t(pg), uint32_t(delta), uint32_t(page));
        bt[j] = page;
        ++j;
      }
      delta += L;
    }
    doc_blocks[b] = j;
    if (uint64_t(delta) >= kMaxDelta) return fail(LAZY_ERANGE, "offset %lld >= 2^24", (long long)delta);
    q_start[b] = int32_t(delta);
    const int nq = q_page_off[b + 1] - q_page_off[b];
    if (nq < 0 || q_len[b] < 0) return fail(LAZY_EINVAL, "bad query segment of request %d", b);
    if (int64_t(nq) * kPage < q_len[b]) return fail(LAZY_EINVAL, "query segment of request %d lacks pages", b);
    if (uint64_t(nq) > kMaxPg) return fail(LAZY_ERANGE, "query segment longer than %d pages", int(kMaxPg));
    for (int pg = 0; pg < nq; ++pg) {
      if (j >= max_blocks) return fail(LAZY_ERANGE, "request %d needs more than max_blocks=%d", b, max_blocks);
      const int32_t page = q_pages[q_page_off[b] + pg];
      if (page < 0 || uint64_t(page) >= kMaxPage) return fail(LAZY_ERANGE, "page id %d out of range", page);
      mw[j] = pack(kPage, uint32_t(pg), uint32_t(delta), uint32_t(page));
      bt[j] = page;
      ++j;
    }
    if (delta + q_len[b] >= int64_t(1) << 31) return fail(LAZY_ERANGE, "sequence too long");
    seq_len[b] = int32_t(delta + q_len[b]);
  }
  return LAZY_OK;
}
