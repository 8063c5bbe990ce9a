// topk_noalloc.cu -- ddt_topk_logprobs_noalloc: the a1 top-K kernel with its
// scratch in one fixed device array instead of a context's workspace, for
// callers that may not allocate device memory (see include/ddt.h).
//
// The array below is part of this library's device image: every GPU that
// loads libddt.so holds it until the process exits. Host code never uses its
// name as a pointer (on the host it is only a stand-in for the symbol); the
// device address comes from cudaGetSymbolAddress, looked up on every call in
// the calling thread's current context, and is passed to the kernel. A
// lookup per call keeps the address right for whatever context is current
// (the primary context, one made with cuCtxCreate, or a new context after a
// device reset); once the library's module is loaded in that context the
// lookup is a table read.
#include <stdint.h>

#include "ddt_internal.h"

namespace {

// scratch layout (byte offsets, each 256-aligned): the status word, per
// (row, chunk) each warp's (max, sum of exp), per row group its max as a
// 16-bit ordered key, and per warp its Q largest keys. With Q as a1 picks it,
// a row's warps keep at most 32 * chunks + 2K + 16 * chunks keys.
constexpr size_t NA_STATUS = 0;
constexpr size_t NA_MS = 256;
constexpr size_t NA_GKEY =
    NA_MS + sizeof(float2) * (TOPK_THREADS / 32) * DDT_NOALLOC_MAX_ROW_CHUNKS;
constexpr size_t NA_WTOP = NA_GKEY + sizeof(uint16_t) * TOPK_THREADS * DDT_NOALLOC_MAX_ROW_CHUNKS;
constexpr size_t NA_WTOP_KEYS =
    48 * (size_t)DDT_NOALLOC_MAX_ROW_CHUNKS + 2 * (size_t)DDT_MAX_K * DDT_NOALLOC_MAX_ROWS;
constexpr size_t NA_BYTES = NA_WTOP + sizeof(uint16_t) * NA_WTOP_KEYS;
static_assert(NA_MS % 256 == 0 && NA_GKEY % 256 == 0 && NA_WTOP % 256 == 0, "alignment");

}  // namespace

// the scratch itself: file scope, fixed size (about 22 MB)
static __device__ __align__(256) unsigned char g_topk_scratch[NA_BYTES];

extern "C" ddt_status ddt_topk_logprobs_noalloc(const void *draft_logits, int32_t draft_dtype,
                                                int32_t rows, int32_t V, int32_t K, float *top_lp,
                                                int32_t *top_ids, void *stream)
{
    // ---- sizes and pointers first: nothing is enqueued on a rejection
    if (draft_dtype != DDT_BF16 && draft_dtype != DDT_F32)
        return DDT_EINVAL;
    if (rows < 0 || V < 1 || K < 1 || K > V)
        return DDT_EINVAL;
    if (rows == 0)
        return DDT_OK;
    if (draft_logits == nullptr || top_lp == nullptr || top_ids == nullptr ||
        ((uintptr_t)draft_logits & 15u) != 0 || ((uintptr_t)top_lp & 3u) != 0 ||
        ((uintptr_t)top_ids & 3u) != 0)
        return DDT_EINVAL;
    const int chunk = topk_chunk_elems(draft_dtype);
    const int64_t nch = ((int64_t)V + chunk - 1) / chunk;
    if (K > DDT_MAX_K || nch * K > TOPK_CAND_CAP || nch > TOPK_MAX_CHUNKS ||
        rows > DDT_NOALLOC_MAX_ROWS ||
        (int64_t)rows * nch > DDT_NOALLOC_MAX_ROW_CHUNKS)
        return DDT_EUNSUPPORTED;

    // ---- the array's device address in the current context (the first call
    // in a context may load the library's module there, which stream capture
    // does not allow: make that call before any capture)
    void *p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_topk_scratch);
    if (e != cudaSuccess) {
        ddt_note_cuda_error((int)e);
        return DDT_ECUDA;
    }
    unsigned char *base = (unsigned char *)p;
    int dev = 0, num_sms = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) {
        ddt_note_cuda_error((int)e);
        return DDT_ECUDA;
    }

    // ---- the array keeps the previous call's contents: every slot this call
    // reads is written by this call first, except the status word, cleared here
    cudaStream_t s = (cudaStream_t)stream;
    e = cudaMemsetAsync(base + NA_STATUS, 0, sizeof(int32_t), s);
    if (e == cudaSuccess)
        e = launch_topk_scratch(draft_logits, draft_dtype, rows, V, K, (int)nch, num_sms,
                                (uint16_t *)(base + NA_GKEY), (uint16_t *)(base + NA_WTOP),
                                (float2 *)(base + NA_MS), top_lp, top_ids,
                                (int32_t *)(base + NA_STATUS), s);
    if (e != cudaSuccess) {
        ddt_note_cuda_error((int)e);
        return DDT_ECUDA;
    }
    return DDT_OK;
}
