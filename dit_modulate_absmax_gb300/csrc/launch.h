// launch.h -- internal launchers behind the C ABI (not exported).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "h3fp4.h"

namespace h3fp4 {

// Row ranges of the modulation segments, passed to kernels by value.
struct SegTable {
    int32_t off[H3FP4_MAX_SEGMENTS + 1];
    int32_t nseg;
};

// Multiprocessor count of the current device (cached per device).
int sm_count();

cudaError_t launch_modulate_absmax(const uint16_t *x, int64_t ldx, int64_t m, int64_t d,
                                   const uint16_t *shift, const uint16_t *scale, int64_t ld_mod,
                                   const SegTable &seg, float *ts, uint32_t *scratch, cudaStream_t st);

cudaError_t launch_modulate_pack(const uint16_t *x, int64_t ldx, int64_t m, int64_t m_pad, int64_t d,
                                 const uint16_t *shift, const uint16_t *scale, int64_t ld_mod,
                                 const SegTable &seg, const float *ts, uint8_t *qdata, uint8_t *sf,
                                 cudaStream_t st);

cudaError_t launch_swiglu_pack(const uint16_t *gate, int64_t ldg, const uint16_t *up, int64_t ldu,
                               int64_t m, int64_t m_pad, int64_t f, float *ts, uint32_t *scratch,
                               uint8_t *qdata, uint8_t *sf, uint16_t *h, cudaStream_t st);

cudaError_t launch_modulate_produce(const uint16_t *x, int64_t ldx, int64_t m, int64_t m_pad, int64_t d,
                                    const uint16_t *shift, const uint16_t *scale, int64_t ld_mod, const SegTable &seg,
                                    float *ts, uint32_t *scratch, uint8_t *qdata, uint8_t *sf, cudaStream_t st);

cudaError_t read_producer_error(uint32_t *code);

cudaError_t launch_quantize_pack(const uint16_t *x, int64_t ldx, int64_t m, int64_t m_pad, int64_t d,
                                 float *ts, uint32_t *scratch, uint8_t *qdata, uint8_t *sf, cudaStream_t st);

cudaError_t launch_swizzle_scales(const uint8_t *src, int64_t rows, int64_t cols, int64_t ld,
                                  uint8_t *dst, cudaStream_t st);

// Gated residual epilogue of the GEMM: out = RN_bf16(residual + RN_bf16(gate_s * c)),
// gate [nseg, n] bf16 selected by the row segments.
struct GatedArgs {
    const uint16_t *gate;
    int64_t ld_gate;
    SegTable seg;
    const void *residual;
    int64_t ldr;
};

h3fp4_status launch_gemm(const uint8_t *a_q, const uint8_t *a_sf, const float *a_ts, const uint8_t *b_q,
                         const uint8_t *b_sf, const float *b_ts, uint16_t *c, int64_t ldc, int64_t m,
                         int64_t m_pad, int64_t n, int64_t k, const h3fp4_gemm_config &cfg, const GatedArgs *gated,
                         cudaStream_t st);

// Failure detection (diagnostics, not the hot path): the default GEMM with its
// operand loads withheld, so that every consumer wait runs out after wait_ns;
// the cooperative plain producer with a grid-barrier arrival target the grid
// cannot meet and a barrier limit of wait_ns.  Outputs are left untouched; the
// kernels record device error bits and return.
h3fp4_status launch_gemm_wait_timeout(const uint8_t *a_q, const uint8_t *a_sf, const float *a_ts,
                                      const uint8_t *b_q, const uint8_t *b_sf, const float *b_ts, uint16_t *c,
                                      int64_t ldc, int64_t m, int64_t m_pad, int64_t n, int64_t k, uint64_t wait_ns,
                                      cudaStream_t st);
cudaError_t launch_quantize_pack_barrier_timeout(const uint16_t *x, int64_t ldx, int64_t m, int64_t m_pad,
                                                int64_t d, float *ts, uint32_t *scratch, uint8_t *qdata, uint8_t *sf,
                                                uint64_t wait_ns, cudaStream_t st);

h3fp4_status read_device_error(uint32_t *code);

}  // namespace h3fp4
