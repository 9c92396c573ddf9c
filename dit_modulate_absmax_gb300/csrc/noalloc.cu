// noalloc.cu -- h3fp4_swiglu_pack_noalloc: the SwiGLU producer with its
// scratch in library-owned static device memory, for callers that cannot
// allocate device memory themselves.
//
// h3fp4_swiglu_pack needs two scratch words (the global absmax and a CTA
// counter) and, to evaluate silu only once, an [m, f] bf16 workspace for h.
// Some callers have no device allocator at hand when they call in: a plugin
// running inside another framework's operator, or a serving loop that must
// not allocate after warm-up.  This entry point takes the same inputs and
// outputs but keeps both scratch areas in one file-scope static __device__
// array of fixed size, so it calls no cudaMalloc, no cudaFree and no
// allocating library routine.
//
// Set-up: the array's device address is looked up once per device (with
// that device current) by cudaGetSymbolAddress on the first call made on it;
// that first call may also load this file's device module, so it should come
// before any stream capture.  The address is kept for the life of the
// process's context on that device: a caller that destroys the context
// (cudaDeviceReset) must not call this entry point again in that process.
//
// Sharing: every call uses the same array and it keeps the last call's
// contents.  The two counter words are cleared on the stream by every call;
// h is fully rewritten by pass 1 before pass 2 reads it.  Calls whose GPU
// work overlaps (different streams, or different host threads, on the same
// device) race on the array and must be serialised by the caller.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "h3fp4.h"
#include "launch.h"

namespace {

constexpr int64_t kCounterBytes = 256;                           // 2 words used, padded for alignment
constexpr int64_t kMaxH = H3FP4_NOALLOC_MAX_ELEMENTS;            // bf16 elements of h
static __device__ __align__(256) uint8_t g_noalloc_scratch[kCounterBytes + 2 * kMaxH];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_addr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device (looked up once).
h3fp4_status scratch_address(void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return H3FP4_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices)
        return H3FP4_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_addr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
            return H3FP4_ERR_CUDA;
        g_addr[dev] = p;
    }
    *out = g_addr[dev];
    return H3FP4_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" h3fp4_status h3fp4_swiglu_pack_noalloc(const void *gate_bf16, int64_t ldg, const void *up_bf16,
                                                  int64_t ldu, int64_t m, int64_t m_pad, int64_t f,
                                                  float *tensor_scale, uint8_t *qdata, uint8_t *sfa, void *stream)
{
    if (((gate_bf16 == nullptr || up_bf16 == nullptr) && m != 0) || tensor_scale == nullptr || qdata == nullptr ||
        sfa == nullptr)
        return H3FP4_ERR_NULL;
    if (m < 0 || m > INT32_MAX || f <= 0 || f % 256 != 0 || f > (int64_t(1) << 24) || ldg < f || ldu < f ||
        m_pad < m || m_pad % 16 != 0 || m_pad > INT32_MAX)
        return H3FP4_ERR_SHAPE;
    if (m * f > kMaxH)
        return H3FP4_ERR_SHAPE;  // h would not fit the static workspace
    if (!aligned16(gate_bf16) || !aligned16(up_bf16) || ldg % 8 != 0 || ldu % 8 != 0 || !aligned16(qdata) ||
        !aligned16(sfa))
        return H3FP4_ERR_ALIGN;
    void *base = nullptr;
    const h3fp4_status s = scratch_address(&base);
    if (s != H3FP4_OK)
        return s;
    uint32_t *counters = static_cast<uint32_t *>(base);
    uint16_t *h = reinterpret_cast<uint16_t *>(static_cast<uint8_t *>(base) + kCounterBytes);
    const cudaError_t e = h3fp4::launch_swiglu_pack(
        static_cast<const uint16_t *>(gate_bf16), ldg, static_cast<const uint16_t *>(up_bf16), ldu, m, m_pad, f,
        tensor_scale, counters, qdata, sfa, h, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? H3FP4_OK : H3FP4_ERR_CUDA;
}
