// api.cu -- the extern "C" entry points declared in include/h3fp4.h.
//
// Each entry point checks its arguments on the host (null pointers, 16-byte
// alignment, leading dimensions, shape multiples, segment table) and only then
// enqueues its kernels; a failed check enqueues nothing.
#include <cuda_runtime.h>

#include <cstdint>

#include "h3fp4.h"
#include "launch.h"

#ifndef H3FP4_VERSION
#define H3FP4_VERSION "0.1.0"
#endif
#define H3FP4_STR2(x) #x
#define H3FP4_STR(x) H3FP4_STR2(x)

namespace {

using h3fp4::SegTable;

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

cudaStream_t as_stream(void *s) { return static_cast<cudaStream_t>(s); }

h3fp4_status from_cuda(cudaError_t e) { return e == cudaSuccess ? H3FP4_OK : H3FP4_ERR_CUDA; }

// Fills `t` from the host offsets; checks 0 = off[0] <= ... <= off[nseg] = m.
h3fp4_status make_segments(const int32_t *off, int32_t nseg, int64_t m, SegTable *t)
{
    if (off == nullptr)
        return H3FP4_ERR_NULL;
    if (nseg < 1 || nseg > H3FP4_MAX_SEGMENTS)
        return H3FP4_ERR_SHAPE;
    if (off[0] != 0 || static_cast<int64_t>(off[nseg]) != m)
        return H3FP4_ERR_SHAPE;
    for (int32_t s = 0; s < nseg; ++s)
        if (off[s + 1] < off[s])
            return H3FP4_ERR_SHAPE;
    for (int32_t s = 0; s <= H3FP4_MAX_SEGMENTS; ++s)
        t->off[s] = s <= nseg ? off[s] : off[nseg];
    t->nseg = nseg;
    return H3FP4_OK;
}

// Shared checks of the modulation producer's inputs.
// x may be NULL when m == 0 (nothing is read from it).
h3fp4_status check_modulate(const void *x, int64_t ldx, int64_t m, int64_t d, const void *shift,
                            const void *scale, int64_t ld_mod)
{
    if ((x == nullptr && m != 0) || shift == nullptr || scale == nullptr)
        return H3FP4_ERR_NULL;
    if (m < 0 || m > INT32_MAX || d <= 0 || d % 256 != 0 || d > (int64_t(1) << 24))
        return H3FP4_ERR_SHAPE;
    if (ldx < d || ld_mod < d)
        return H3FP4_ERR_SHAPE;
    if (!aligned16(x) || !aligned16(shift) || !aligned16(scale) || ldx % 8 != 0 || ld_mod % 8 != 0)
        return H3FP4_ERR_ALIGN;
    return H3FP4_OK;
}

h3fp4_status check_pack_outputs(int64_t m, int64_t m_pad, const void *qdata, const void *sf)
{
    if (qdata == nullptr || sf == nullptr)
        return H3FP4_ERR_NULL;
    if (m_pad < m || m_pad % 16 != 0 || m_pad > INT32_MAX)   // the GEMM's descriptor M: a multiple of 16
        return H3FP4_ERR_SHAPE;
    if (!aligned16(qdata) || !aligned16(sf))
        return H3FP4_ERR_ALIGN;
    return H3FP4_OK;
}

}  // namespace

extern "C" {

h3fp4_status h3fp4_modulate_absmax(const void *x_bf16, int64_t ldx, int64_t m, int64_t d, const void *shift_bf16,
                                   const void *scale_bf16, int64_t ld_mod, const int32_t *seg_row_offsets,
                                   int32_t nseg, float *tensor_scale, uint32_t *scratch, void *stream)
{
    h3fp4_status s = check_modulate(x_bf16, ldx, m, d, shift_bf16, scale_bf16, ld_mod);
    if (s != H3FP4_OK)
        return s;
    if (tensor_scale == nullptr || scratch == nullptr)
        return H3FP4_ERR_NULL;
    SegTable seg;
    if ((s = make_segments(seg_row_offsets, nseg, m, &seg)) != H3FP4_OK)
        return s;
    return from_cuda(h3fp4::launch_modulate_absmax(
        static_cast<const uint16_t *>(x_bf16), ldx, m, d, static_cast<const uint16_t *>(shift_bf16),
        static_cast<const uint16_t *>(scale_bf16), ld_mod, seg, tensor_scale, scratch, as_stream(stream)));
}

h3fp4_status h3fp4_modulate_pack(const void *x_bf16, int64_t ldx, int64_t m, int64_t m_pad, int64_t d,
                                 const void *shift_bf16, const void *scale_bf16, int64_t ld_mod,
                                 const int32_t *seg_row_offsets, int32_t nseg, const float *tensor_scale,
                                 uint8_t *qdata, uint8_t *sfa, void *stream)
{
    h3fp4_status s = check_modulate(x_bf16, ldx, m, d, shift_bf16, scale_bf16, ld_mod);
    if (s != H3FP4_OK)
        return s;
    if (tensor_scale == nullptr)
        return H3FP4_ERR_NULL;
    if ((s = check_pack_outputs(m, m_pad, qdata, sfa)) != H3FP4_OK)
        return s;
    SegTable seg;
    if ((s = make_segments(seg_row_offsets, nseg, m, &seg)) != H3FP4_OK)
        return s;
    return from_cuda(h3fp4::launch_modulate_pack(
        static_cast<const uint16_t *>(x_bf16), ldx, m, m_pad, d, static_cast<const uint16_t *>(shift_bf16),
        static_cast<const uint16_t *>(scale_bf16), ld_mod, seg, tensor_scale, qdata, sfa, as_stream(stream)));
}

h3fp4_status h3fp4_modulate_produce(const void *x_bf16, int64_t ldx, int64_t m, int64_t m_pad, int64_t d,
                                    const void *shift_bf16, const void *scale_bf16, int64_t ld_mod,
                                    const int32_t *seg_row_offsets, int32_t nseg, float *tensor_scale,
                                    uint32_t *scratch, uint8_t *qdata, uint8_t *sfa, void *stream)
{
    h3fp4_status s = check_modulate(x_bf16, ldx, m, d, shift_bf16, scale_bf16, ld_mod);
    if (s != H3FP4_OK)
        return s;
    if (tensor_scale == nullptr || scratch == nullptr)
        return H3FP4_ERR_NULL;
    if ((s = check_pack_outputs(m, m_pad, qdata, sfa)) != H3FP4_OK)
        return s;
    SegTable seg;
    if ((s = make_segments(seg_row_offsets, nseg, m, &seg)) != H3FP4_OK)
        return s;
    return from_cuda(h3fp4::launch_modulate_produce(
        static_cast<const uint16_t *>(x_bf16), ldx, m, m_pad, d, static_cast<const uint16_t *>(shift_bf16),
        static_cast<const uint16_t *>(scale_bf16), ld_mod, seg, tensor_scale, scratch, qdata, sfa, as_stream(stream)));
}

h3fp4_status h3fp4_swiglu_pack(const void *gate_bf16, int64_t ldg, const void *up_bf16, int64_t ldu, int64_t m,
                               int64_t m_pad, int64_t f, float *tensor_scale, uint32_t *scratch, uint8_t *qdata,
                               uint8_t *sfa, void *h_workspace, void *stream)
{
    if (((gate_bf16 == nullptr || up_bf16 == nullptr) && m != 0) || tensor_scale == nullptr || scratch == nullptr)
        return H3FP4_ERR_NULL;
    if (m < 0 || m > INT32_MAX || f <= 0 || f % 256 != 0 || f > (int64_t(1) << 24) || ldg < f || ldu < f)
        return H3FP4_ERR_SHAPE;
    if (!aligned16(gate_bf16) || !aligned16(up_bf16) || ldg % 8 != 0 || ldu % 8 != 0 ||
        (h_workspace != nullptr && !aligned16(h_workspace)))
        return H3FP4_ERR_ALIGN;
    h3fp4_status s = check_pack_outputs(m, m_pad, qdata, sfa);
    if (s != H3FP4_OK)
        return s;
    return from_cuda(h3fp4::launch_swiglu_pack(
        static_cast<const uint16_t *>(gate_bf16), ldg, static_cast<const uint16_t *>(up_bf16), ldu, m, m_pad, f,
        tensor_scale, scratch, qdata, sfa, static_cast<uint16_t *>(h_workspace), as_stream(stream)));
}

h3fp4_status h3fp4_quantize_pack(const void *x_bf16, int64_t ldx, int64_t m, int64_t m_pad, int64_t d,
                                 float *tensor_scale, uint32_t *scratch, uint8_t *qdata, uint8_t *sfa, void *stream)
{
    if ((x_bf16 == nullptr && m != 0) || tensor_scale == nullptr || scratch == nullptr)
        return H3FP4_ERR_NULL;
    if (m < 0 || m > INT32_MAX || d <= 0 || d % 256 != 0 || d > (int64_t(1) << 24) || ldx < d)
        return H3FP4_ERR_SHAPE;
    if (!aligned16(x_bf16) || ldx % 8 != 0)
        return H3FP4_ERR_ALIGN;
    h3fp4_status s = check_pack_outputs(m, m_pad, qdata, sfa);
    if (s != H3FP4_OK)
        return s;
    return from_cuda(h3fp4::launch_quantize_pack(static_cast<const uint16_t *>(x_bf16), ldx, m, m_pad, d,
                                                 tensor_scale, scratch, qdata, sfa, as_stream(stream)));
}

namespace {

// Checks shared by both GEMM entry points; fills `c` with the configuration.
h3fp4_status check_gemm(const uint8_t *a_q, const uint8_t *a_sf, const float *a_tensor_scale, const uint8_t *b_q,
                        const uint8_t *b_sf, const float *b_tensor_scale, const void *c_bf16, int64_t ldc, int64_t m,
                        int64_t m_pad, int64_t n, int64_t k, const h3fp4_gemm_config *cfg, h3fp4_gemm_config *c)
{
    if (a_q == nullptr || a_sf == nullptr || a_tensor_scale == nullptr || b_q == nullptr || b_sf == nullptr ||
        b_tensor_scale == nullptr || (c_bf16 == nullptr && m != 0 && n != 0))
        return H3FP4_ERR_NULL;
    if (m < 0 || m > m_pad || m_pad % 16 != 0 || m_pad > INT32_MAX || n < 0 || n % 128 != 0 || n > INT32_MAX ||
        k <= 0 || k % 256 != 0 || k > (int64_t(1) << 24) || ldc < n)
        return H3FP4_ERR_SHAPE;
    if (!aligned16(a_q) || !aligned16(a_sf) || !aligned16(b_q) || !aligned16(b_sf) || !aligned16(c_bf16) ||
        ldc % 8 != 0)
        return H3FP4_ERR_ALIGN;
    *c = h3fp4_gemm_config{0, 0, 0, 0};
    if (cfg != nullptr) {
        *c = *cfg;
        if (c->n_group < 0 || c->stages != 0 || (c->cta_pair != 0 && c->cta_pair != 1 && c->cta_pair != 4) ||
            c->reserved != 0)
            return H3FP4_ERR_UNSUPPORTED;
    }
    return H3FP4_OK;
}

}  // namespace

h3fp4_status h3fp4_gemm(const uint8_t *a_q, const uint8_t *a_sf, const float *a_tensor_scale, const uint8_t *b_q,
                        const uint8_t *b_sf, const float *b_tensor_scale, void *c_bf16, int64_t ldc, int64_t m,
                        int64_t m_pad, int64_t n, int64_t k, const h3fp4_gemm_config *cfg, void *stream)
{
    h3fp4_gemm_config c;
    h3fp4_status s = check_gemm(a_q, a_sf, a_tensor_scale, b_q, b_sf, b_tensor_scale, c_bf16, ldc, m, m_pad, n, k, cfg, &c);
    if (s != H3FP4_OK)
        return s;
    return h3fp4::launch_gemm(a_q, a_sf, a_tensor_scale, b_q, b_sf, b_tensor_scale,
                              static_cast<uint16_t *>(c_bf16), ldc, m, m_pad, n, k, c, nullptr, as_stream(stream));
}

h3fp4_status h3fp4_gemm_gated_residual(const uint8_t *a_q, const uint8_t *a_sf, const float *a_tensor_scale,
                                       const uint8_t *b_q, const uint8_t *b_sf, const float *b_tensor_scale,
                                       const void *gate_bf16, int64_t ld_gate, const int32_t *seg_row_offsets,
                                       int32_t nseg, const void *residual_bf16, int64_t ldr, void *out_bf16,
                                       int64_t ldo, int64_t m, int64_t m_pad, int64_t n, int64_t k,
                                       const h3fp4_gemm_config *cfg, void *stream)
{
    h3fp4_gemm_config c;
    h3fp4_status s = check_gemm(a_q, a_sf, a_tensor_scale, b_q, b_sf, b_tensor_scale, out_bf16, ldo, m, m_pad, n, k,
                                cfg, &c);
    if (s != H3FP4_OK)
        return s;
    const bool rows = m != 0 && n != 0;
    if (rows && (gate_bf16 == nullptr || residual_bf16 == nullptr))
        return H3FP4_ERR_NULL;
    if (ld_gate < n || ldr < n)
        return H3FP4_ERR_SHAPE;
    if (!aligned16(gate_bf16) || !aligned16(residual_bf16) || ld_gate % 8 != 0 || ldr % 8 != 0)
        return H3FP4_ERR_ALIGN;
    SegTable seg;
    if ((s = make_segments(seg_row_offsets, nseg, m, &seg)) != H3FP4_OK)
        return s;
    if (rows) {   // the output either is the residual (same leading dimension) or does not overlap it
        const char *o = static_cast<const char *>(out_bf16), *r = static_cast<const char *>(residual_bf16);
        const int64_t ob = ((m - 1) * ldo + n) * 2, rb = ((m - 1) * ldr + n) * 2;
        const bool same = o == r && ldo == ldr;
        if (!same && o < r + rb && r < o + ob)
            return H3FP4_ERR_UNSUPPORTED;
    }
    h3fp4::GatedArgs g{static_cast<const uint16_t *>(gate_bf16), ld_gate, seg, residual_bf16, ldr};
    return h3fp4::launch_gemm(a_q, a_sf, a_tensor_scale, b_q, b_sf, b_tensor_scale, static_cast<uint16_t *>(out_bf16),
                              ldo, m, m_pad, n, k, c, &g, as_stream(stream));
}

h3fp4_status h3fp4_swizzle_scales(const uint8_t *sf_logical, int64_t rows, int64_t cols, int64_t ld,
                                  uint8_t *sf_out, void *stream)
{
    if (sf_logical == nullptr || sf_out == nullptr)
        return H3FP4_ERR_NULL;
    if (rows < 0 || cols <= 0 || cols % 4 != 0 || ld < cols || rows > INT32_MAX)
        return H3FP4_ERR_SHAPE;
    if (!aligned16(sf_out))
        return H3FP4_ERR_ALIGN;
    return from_cuda(h3fp4::launch_swizzle_scales(sf_logical, rows, cols, ld, sf_out, as_stream(stream)));
}

h3fp4_status h3fp4_diag_producer_barrier_timeout(const void *x_bf16, int64_t ldx, int64_t m, int64_t m_pad,
                                                 int64_t d, float *tensor_scale, uint32_t *scratch, uint8_t *qdata,
                                                 uint8_t *sfa, uint32_t limit_us, void *stream)
{
    if ((x_bf16 == nullptr && m != 0) || tensor_scale == nullptr || scratch == nullptr)
        return H3FP4_ERR_NULL;
    if (m < 0 || m > INT32_MAX || d <= 0 || d % 256 != 0 || d > (int64_t(1) << 24) || ldx < d || limit_us == 0 ||
        limit_us > 2000000u)
        return H3FP4_ERR_SHAPE;
    if (!aligned16(x_bf16) || ldx % 8 != 0)
        return H3FP4_ERR_ALIGN;
    h3fp4_status s = check_pack_outputs(m, m_pad, qdata, sfa);
    if (s != H3FP4_OK)
        return s;
    return from_cuda(h3fp4::launch_quantize_pack_barrier_timeout(
        static_cast<const uint16_t *>(x_bf16), ldx, m, m_pad, d, tensor_scale, scratch, qdata, sfa,
        static_cast<uint64_t>(limit_us) * 1000u, as_stream(stream)));
}

h3fp4_status h3fp4_diag_gemm_wait_timeout(const uint8_t *a_q, const uint8_t *a_sf, const float *a_tensor_scale,
                                          const uint8_t *b_q, const uint8_t *b_sf, const float *b_tensor_scale,
                                          void *c_bf16, int64_t ldc, int64_t m, int64_t m_pad, int64_t n, int64_t k,
                                          uint32_t limit_us, void *stream)
{
    h3fp4_gemm_config c;
    h3fp4_status s = check_gemm(a_q, a_sf, a_tensor_scale, b_q, b_sf, b_tensor_scale, c_bf16, ldc, m, m_pad, n, k,
                                nullptr, &c);
    if (s != H3FP4_OK)
        return s;
    if (limit_us == 0 || limit_us > 2000000u)
        return H3FP4_ERR_SHAPE;
    return h3fp4::launch_gemm_wait_timeout(a_q, a_sf, a_tensor_scale, b_q, b_sf, b_tensor_scale,
                                           static_cast<uint16_t *>(c_bf16), ldc, m, m_pad, n, k,
                                           static_cast<uint64_t>(limit_us) * 1000u, as_stream(stream));
}

h3fp4_status h3fp4_device_error(uint32_t *code)
{
    if (code == nullptr)
        return H3FP4_ERR_NULL;
    return h3fp4::read_device_error(code);
}

const char *h3fp4_status_string(h3fp4_status status)
{
    switch (status) {
    case H3FP4_OK: return "ok";
    case H3FP4_ERR_NULL: return "null pointer";
    case H3FP4_ERR_ALIGN: return "misaligned pointer or leading dimension";
    case H3FP4_ERR_SHAPE: return "invalid shape";
    case H3FP4_ERR_UNSUPPORTED: return "unsupported configuration";
    case H3FP4_ERR_CUDA: return "CUDA error";
    case H3FP4_ERR_DEVICE: return "device-side error";
    }
    return "unknown status";
}

const char *h3fp4_build_info(void)
{
    return "h3fp4 " H3FP4_VERSION " sm_103a (nvcc " H3FP4_STR(__CUDACC_VER_MAJOR__) "." H3FP4_STR(
        __CUDACC_VER_MINOR__) "." H3FP4_STR(__CUDACC_VER_BUILD__) ")";
}

}  // extern "C"
