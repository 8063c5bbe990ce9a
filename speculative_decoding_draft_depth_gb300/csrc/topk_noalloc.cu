// topk_noalloc.cu -- ddt_topk_logprobs_noalloc: the a1 top-K kernel with its
// scratch in one fixed device array instead of a context's workspace, for
// callers that may not allocate device memory (see include/ddt.h).
//
// The array below is part of this library's device image: every GPU that
// loads libddt.so holds it until the process exits. Host code never uses its
// name as a pointer (on the host it is only a stand-in for the symbol); the
// device address comes from cudaGetSymbolAddress, looked up once per device
// with that device current, and is passed to the kernel.
#include <mutex>
#include <stdint.h>

#include "ddt_internal.h"

namespace {

// scratch layout (byte offsets, each 256-aligned)
constexpr size_t NA_STATUS = 0;
constexpr size_t NA_CNT = 256;
constexpr size_t NA_MS = NA_CNT + sizeof(unsigned) * DDT_NOALLOC_MAX_ROWS;
constexpr size_t NA_VAL = NA_MS + sizeof(float2) * DDT_NOALLOC_MAX_ROW_CHUNKS;
constexpr size_t NA_IDX = NA_VAL + sizeof(float) * DDT_NOALLOC_MAX_ENTRIES;
constexpr size_t NA_BYTES = NA_IDX + sizeof(int32_t) * DDT_NOALLOC_MAX_ENTRIES;
static_assert(NA_MS % 256 == 0 && NA_VAL % 256 == 0 && NA_IDX % 256 == 0, "alignment");

constexpr int NA_MAX_DEVICES = 64;

std::mutex g_mu;
unsigned char *g_base[NA_MAX_DEVICES];  // device address per device, once looked up

}  // namespace

// the scratch itself: file scope, fixed size (about 8.5 MB)
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
    if (K > DDT_MAX_K || nch * K > TOPK_CAND_CAP || rows > DDT_NOALLOC_MAX_ROWS ||
        (int64_t)rows * nch > DDT_NOALLOC_MAX_ROW_CHUNKS ||
        (int64_t)rows * nch * K > DDT_NOALLOC_MAX_ENTRIES)
        return DDT_EUNSUPPORTED;

    // ---- once per device: the array's device address, with that device current
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        ddt_note_cuda_error((int)e);
        return DDT_ECUDA;
    }
    if (dev < 0 || dev >= NA_MAX_DEVICES)
        return DDT_EUNSUPPORTED;
    unsigned char *base;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if (g_base[dev] == nullptr) {
            void *p = nullptr;
            e = cudaGetSymbolAddress(&p, g_topk_scratch);
            if (e != cudaSuccess) {
                ddt_note_cuda_error((int)e);
                return DDT_ECUDA;
            }
            g_base[dev] = (unsigned char *)p;
        }
        base = g_base[dev];
    }

    // ---- the array keeps the previous call's contents: zero the arrival
    // counters and the status word this call relies on
    cudaStream_t s = (cudaStream_t)stream;
    e = cudaMemsetAsync(base + NA_CNT, 0, sizeof(unsigned) * (size_t)rows, s);
    if (e == cudaSuccess)
        e = cudaMemsetAsync(base + NA_STATUS, 0, sizeof(int32_t), s);
    if (e == cudaSuccess)
        e = launch_topk_scratch(draft_logits, draft_dtype, rows, V, K, (int)nch,
                                (float *)(base + NA_VAL), (int32_t *)(base + NA_IDX),
                                (float2 *)(base + NA_MS), (unsigned *)(base + NA_CNT), top_lp,
                                top_ids, (int32_t *)(base + NA_STATUS), s);
    if (e != cudaSuccess) {
        ddt_note_cuda_error((int)e);
        return DDT_ECUDA;
    }
    return DDT_OK;
}
