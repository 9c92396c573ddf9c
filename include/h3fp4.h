/*
 * h3fp4.h -- C ABI of the GB300 (sm_103a) modulation-fused NVFP4 activation
 * producer and block-scaled NVFP4 GEMM.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every pointer is CALLER-OWNED DEVICE memory unless its comment says
 *    "host".  The library never allocates device memory and keeps no pointer
 *    after the call returns.  A pointer to an array with zero rows (the
 *    activation inputs when m == 0, the GEMM output when m == 0 or n == 0)
 *    may be NULL.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    Every call only enqueues work on that stream and returns; nothing
 *    synchronises the host.  Outputs are valid once the stream reaches them.
 *    The first call of an entry point on a device sets its kernels'
 *    attributes; after that, h3fp4_modulate_absmax, h3fp4_modulate_pack,
 *    h3fp4_swiglu_pack and h3fp4_gemm may be captured into a CUDA graph and
 *    replayed (the captured calls keep their pointers; new inputs are copied
 *    into the same buffers).
 *  - Arguments are checked on the host before anything is enqueued.  A failed
 *    check returns an error status and enqueues nothing.  A CUDA launch error
 *    returns H3FP4_ERR_CUDA (the CUDA error itself stays readable with
 *    cudaGetLastError()).  No entry point traps or aborts.
 *  - bf16 tensors are raw IEEE bfloat16 bit patterns (2 bytes), row-major,
 *    with the given leading dimension in ELEMENTS.
 *  - QDATA is packed E2M1, row-major [rows, width/2] bytes, element 2i in the
 *    low nibble of byte i and element 2i+1 in the high nibble.
 *  - Block scales (SFA / SFB) are E4M3 (bias 7, max 448, no infinities), one
 *    per 16 consecutive values of a row, stored in the block-scaled GEMM's
 *    scale layout: the logical [R, C] scale matrix (R = rows rounded up to a
 *    multiple of 128, C = width/16) is cut into 128 x 4 tiles stored
 *    tile-row-major as 512-byte atoms, and inside an atom the scale of row r,
 *    column c sits at byte (r % 32) * 16 + ((r % 128) / 32) * 4 + (c % 4).
 *    A scale buffer for `rows` rows therefore holds ceil(rows/128)*128 * C
 *    bytes.
 *
 * Numerics (fixed encoding rule; the source pages name the quantities but not
 * the reciprocal detail):
 *    y   = RN_bf16(RN_bf16(x * RN_bf16(scale + 1)) + shift)
 *    ts  = RN_f32(amax / 2688)                       (2688 = 6 * 448)
 *    bs  = E4M3_RNE_sat(RN_f32(block_amax / RN_f32(6 * ts)))   (0 if block_amax == 0)
 *    q   = E2M1_RNE_sat(RN_f32(y / RN_f32(dec(bs) * ts)))      (signed 0 if that product is 0)
 *    C   = RN_bf16(RN_f32(ts_a * ts_b) * sum_k a_k b_k)        (FP32 accumulation)
 * Non-finite inputs follow the same formulas in IEEE arithmetic: a NaN makes
 * its block maximum, amax and ts NaN, an infinity makes ts infinite; a NaN
 * quotient encodes as the E4M3 NaN code 0x7F and a NaN scale product, like a
 * zero one, gives zeros with y's signs.  So a tensor holding a NaN or an
 * infinity packs to signed-zero codes with scale 0x7F on its non-zero blocks
 * (0 on blocks whose quotient is 0), and any GEMM over it is NaN.
 */
#ifndef H3FP4_H
#define H3FP4_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define H3FP4_API __attribute__((visibility("default")))
#else
#define H3FP4_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum h3fp4_status {
    H3FP4_OK = 0,
    H3FP4_ERR_NULL = 1,        /* a required pointer is NULL */
    H3FP4_ERR_ALIGN = 2,       /* a pointer or leading dimension breaks the 16-byte rule */
    H3FP4_ERR_SHAPE = 3,       /* a size is negative, too large, or not a required multiple */
    H3FP4_ERR_UNSUPPORTED = 4, /* a configuration the library does not implement */
    H3FP4_ERR_CUDA = 5,        /* a CUDA call failed (see cudaGetLastError) */
    H3FP4_ERR_DEVICE = 6       /* a kernel recorded a device-side error (bounded wait ran out) */
} h3fp4_status;

/* Most modulation segments one call accepts. */
#define H3FP4_MAX_SEGMENTS 16

/*
 * h3fp4_modulate_absmax -- producer pass 1.
 * Source: "NVFP4 Modulation Producer Fusion", Dataflow (prototype step 1) and
 * Exactness Contract; "NVFP4 Streaming Design", Numerical Constraint items 1-2.
 *
 * Modulates every logical row of x (row r uses segment s, the one with
 * seg_row_offsets[s] <= r < seg_row_offsets[s+1]) without storing the result,
 * reduces one exact global max |y| over rows [0, m), and writes the FP32
 * tensor scale RN_f32(amax / 2688) to *tensor_scale.  A NaN anywhere in y
 * makes the tensor scale NaN.
 *
 *   x_bf16          [m, d] bf16, leading dimension ldx (>= d, multiple of 8), 16-byte aligned
 *   shift_bf16      [nseg, d] bf16, leading dimension ld_mod (>= d, multiple of 8), 16-byte aligned
 *   scale_bf16      [nseg, d] bf16, same layout as shift
 *   seg_row_offsets HOST array of nseg + 1 int32: 0 = off[0] <= off[1] <= ... <= off[nseg] = m
 *   nseg            1 .. H3FP4_MAX_SEGMENTS
 *   tensor_scale    1 float (output)
 *   scratch         2 uint32 words of device scratch (contents on entry are ignored; the
 *                   call clears them on the stream).  Two calls that overlap on the GPU
 *                   must not share it.
 *   d               multiple of 256; m >= 0 (m == 0 gives tensor scale 0)
 */
H3FP4_API h3fp4_status h3fp4_modulate_absmax(const void *x_bf16, int64_t ldx, int64_t m, int64_t d,
                                   const void *shift_bf16, const void *scale_bf16, int64_t ld_mod,
                                   const int32_t *seg_row_offsets, int32_t nseg,
                                   float *tensor_scale, uint32_t *scratch, void *stream);

/*
 * h3fp4_modulate_pack -- producer pass 2.
 * Source: "NVFP4 Modulation Producer Fusion", Dataflow (prototype step 2);
 * "NVFP4 Streaming Design", Numerical Constraint items 3-4; "FC2 NVFP4 Library
 * Scheduling", Exact Operation (zero-row padding to the descriptor M).
 *
 * Re-derives y exactly as pass 1 does and writes QDATA and SFA for rows
 * [0, m_pad).  Rows m <= r < m_pad get zero QDATA bytes; every scale of a row
 * r >= m (up to ceil(m_pad/128)*128) is 0.  Every byte of both buffers is
 * written.
 *
 *   tensor_scale  1 float (input, normally the output of pass 1)
 *   qdata         [m_pad, d/2] bytes, 16-byte aligned
 *   sfa           ceil(m_pad/128)*128 * d/16 bytes in the scale layout, 16-byte aligned
 *   m <= m_pad; other arguments as for h3fp4_modulate_absmax.
 */
H3FP4_API h3fp4_status h3fp4_modulate_pack(const void *x_bf16, int64_t ldx, int64_t m, int64_t m_pad,
                                 int64_t d, const void *shift_bf16, const void *scale_bf16,
                                 int64_t ld_mod, const int32_t *seg_row_offsets, int32_t nseg,
                                 const float *tensor_scale, uint8_t *qdata, uint8_t *sfa,
                                 void *stream);

/*
 * h3fp4_modulate_produce -- h3fp4_modulate_absmax followed by
 * h3fp4_modulate_pack in ONE cooperative launch.
 * Source: "NVFP4 Streaming Design", P2 (a single-launch cooperative producer:
 * pass 1 and pass 2 around a grid barrier, with a bounded wait).
 *
 * Same arguments and results as the two calls (tensor_scale is written and
 * also used by the pack).  Every CTA of the co-resident grid reduces its
 * pass-1 tiles, arrives on a grid barrier in `scratch` and packs its pass-2
 * tiles once all have arrived; the barrier gives up after 2 s, reporting
 * bit 8 through h3fp4_device_error instead of hanging.
 */
H3FP4_API h3fp4_status h3fp4_modulate_produce(const void *x_bf16, int64_t ldx, int64_t m, int64_t m_pad,
                                    int64_t d, const void *shift_bf16, const void *scale_bf16,
                                    int64_t ld_mod, const int32_t *seg_row_offsets, int32_t nseg,
                                    float *tensor_scale, uint32_t *scratch, uint8_t *qdata,
                                    uint8_t *sfa, void *stream);

/*
 * h3fp4_swiglu_pack -- SwiGLU-fused producer (both passes, in one cooperative launch).
 * Source: "FC2 NVFP4 Library Scheduling", Exact Operation and Current Baseline
 * (exact BF16 SwiGLU fused into NVFP4 production of the FC2 input).
 *
 * h = RN_bf16(silu_bf16(gate) * up) with silu_bf16 the correctly rounded bf16
 * of g / (1 + e^-g); then the global absmax -> tensor scale and the pack of h,
 * exactly as the modulation producer does for y.
 *
 *   gate_bf16, up_bf16  [m, f] bf16, leading dimensions ldg / ldu (multiples of 8), 16-byte aligned
 *   f                   multiple of 256
 *   tensor_scale        1 float (output)
 *   scratch             2 uint32 words (as for h3fp4_modulate_absmax)
 *   qdata, sfa          as for h3fp4_modulate_pack with d = f
 *   h_workspace         NULL, or [m, f] bf16 (leading dimension f) that pass 1 fills with h
 *                       so that pass 2 reads h instead of recomputing it
 */
H3FP4_API h3fp4_status h3fp4_swiglu_pack(const void *gate_bf16, int64_t ldg, const void *up_bf16,
                               int64_t ldu, int64_t m, int64_t m_pad, int64_t f,
                               float *tensor_scale, uint32_t *scratch, uint8_t *qdata,
                               uint8_t *sfa, void *h_workspace, void *stream);

/*
 * h3fp4_quantize_pack -- NVFP4 producer of an activation that needs no fused
 * transform (both passes, in one cooperative launch).
 * Source: "NVFP4 Modulation Producer Fusion", Change Summary (the same two-pass
 * producer: global absmax -> FP32 tensor scale, then E4M3 block scales and
 * E2M1 codes); "NVFP4 Streaming Design", P0 and P2 (the attention-output
 * projection is one of the four H3 projections, its input quantized by the
 * same rules without the modulation).
 *
 * amax = max |x| over the m logical rows, ts = RN_f32(amax / 2688), then the
 * pack of x exactly as h3fp4_modulate_pack packs y.
 *
 *   x_bf16        [m, d] bf16, leading dimension ldx (multiple of 8), 16-byte aligned
 *   d             multiple of 256
 *   tensor_scale  1 float (output)
 *   scratch       2 uint32 words (as for h3fp4_modulate_absmax)
 *   qdata, sfa    as for h3fp4_modulate_pack
 */
H3FP4_API h3fp4_status h3fp4_quantize_pack(const void *x_bf16, int64_t ldx, int64_t m, int64_t m_pad,
                                 int64_t d, float *tensor_scale, uint32_t *scratch, uint8_t *qdata,
                                 uint8_t *sfa, void *stream);

/* Tuning knobs of the GEMM; pass NULL for the defaults. */
typedef struct h3fp4_gemm_config {
    /* N-group A-tile reuse factor: the persistent schedule walks the output
     * tiles (256 columns wide) in groups of n_group N-tiles x all M-tiles, N
     * fastest, so each A row block serves n_group consecutive output tiles
     * while it is L2-resident (0 = kernel default: the default kernel takes
     * the fewest near-equal groups whose B tiles total at most ~27.5 MB, the
     * others 28; values above the number of N-tiles are clamped). */
    int32_t n_group;
    int32_t stages;    /* reserved, must be 0 (the pipeline depth is fixed per kernel) */
    /* GEMM kernel: 0 = library default (currently 4), 1 = one CTA per 128 x 256 output tile
     * (4-stage ring, scale warps stage the scales in TMEM), 4 = CTA pairs on
     * two SMs per 256 x 256 tile (tcgen05 cta_group::2, each SM loads its own
     * half of A and of B; 5-stage ring) whose leader copies the scales into
     * TMEM with tcgen05.cp from two warps of their own.  Other values:
     * H3FP4_ERR_UNSUPPORTED. */
    int32_t cta_pair;
    int32_t reserved;  /* must be 0 */
} h3fp4_gemm_config;

/*
 * h3fp4_gemm -- block-scaled NVFP4 GEMM with the alpha epilogue.
 * Source: "NVFP4 Streaming Design", Available Foundation (E2M1 A/B, E4M3
 * scales, FP32 accumulation, BF16 output) and P0 (alpha = activation tensor
 * scale x weight tensor scale applied before the BF16 conversion); "FC2 NVFP4
 * Library Scheduling", Exact Operation (row-major activation [M,K] times
 * weight [N,K] to row-major BF16 [M,N], alpha from device pointers, logical
 * rows sliced from the padded descriptor M).
 *
 * C[i, j] = RN_bf16(RN_f32(*a_tensor_scale * *b_tensor_scale) * acc[i, j]),
 * acc = FP32 accumulation over k of e2m1(a) e4m3(sfa) e2m1(b) e4m3(sfb).
 * Only rows i < m and columns j < n are written.
 *
 *   a_q   [m_pad, k/2] bytes (activation QDATA), 16-byte aligned
 *   a_sf  ceil(m_pad/128)*128 * k/16 bytes, scale layout, 16-byte aligned
 *   b_q   [n, k/2] bytes (weight QDATA), 16-byte aligned
 *   b_sf  ceil(n/128)*128 * k/16 bytes, scale layout, 16-byte aligned
 *   a_tensor_scale, b_tensor_scale   1 float each
 *   c_bf16  [m, n] bf16 output with leading dimension ldc (>= n, multiple of 8), 16-byte aligned
 *   k multiple of 256; n multiple of 128; 0 <= m <= m_pad; m_pad multiple of 16
 */
H3FP4_API h3fp4_status h3fp4_gemm(const uint8_t *a_q, const uint8_t *a_sf, const float *a_tensor_scale,
                        const uint8_t *b_q, const uint8_t *b_sf, const float *b_tensor_scale,
                        void *c_bf16, int64_t ldc, int64_t m, int64_t m_pad, int64_t n, int64_t k,
                        const h3fp4_gemm_config *cfg, void *stream);

/*
 * h3fp4_gemm_gated_residual -- h3fp4_gemm with the gated residual epilogue.
 * Source: "NVFP4 Streaming Design", P4: Exact Epilogue (after the owned GEMM,
 * the explicit BF16 conversion, gate multiply, residual add and final BF16
 * rounding sequence), for the projections whose output is added to the
 * residual stream through an AdaLN gate (attention output, FC2).
 *
 * out[i, j] = RN_bf16(residual[i, j] + RN_bf16(gate[s(i), j] * c[i, j]))
 * with c[i, j] the value h3fp4_gemm would write and s(i) the segment of row i
 * (seg_row_offsets as for h3fp4_modulate_absmax: host array of nseg + 1
 * non-decreasing offsets, [0] = 0, [nseg] = m).  Only rows i < m and columns
 * j < n are written.
 *
 *   gate_bf16      [nseg, n] bf16, leading dimension ld_gate (>= n, multiple of 8), 16-byte aligned
 *   residual_bf16  [m, n] bf16, leading dimension ldr (>= n, multiple of 8), 16-byte aligned
 *   out_bf16       [m, n] bf16, leading dimension ldo; either the residual itself (same pointer and
 *                  leading dimension: updated in place) or not overlapping it (else H3FP4_ERR_UNSUPPORTED)
 *   other arguments as for h3fp4_gemm
 */
H3FP4_API h3fp4_status h3fp4_gemm_gated_residual(
    const uint8_t *a_q, const uint8_t *a_sf, const float *a_tensor_scale, const uint8_t *b_q, const uint8_t *b_sf,
    const float *b_tensor_scale, const void *gate_bf16, int64_t ld_gate, const int32_t *seg_row_offsets, int32_t nseg,
    const void *residual_bf16, int64_t ldr, void *out_bf16, int64_t ldo, int64_t m, int64_t m_pad, int64_t n,
    int64_t k, const h3fp4_gemm_config *cfg, void *stream);

/*
 * h3fp4_swizzle_scales -- helper for preparing weights: copies a LOGICAL
 * row-major E4M3 scale matrix [rows, cols] (leading dimension ld bytes) into
 * the scale layout above, padding rows up to a multiple of 128 with zeros.
 * Not part of the hot path (weights are prepared once).
 *
 *   cols multiple of 4; out holds ceil(rows/128)*128 * cols bytes, 16-byte aligned
 */
H3FP4_API h3fp4_status h3fp4_swizzle_scales(const uint8_t *sf_logical, int64_t rows, int64_t cols,
                                  int64_t ld, uint8_t *sf_out, void *stream);

/*
 * h3fp4_swiglu_pack_noalloc -- h3fp4_swiglu_pack for callers that cannot
 * allocate device memory.  No counterpart on the source pages.
 *
 * Some callers have no device allocator at hand when they call in (a plugin
 * running inside another framework's operator, a serving loop that must not
 * allocate after warm-up), so they cannot pass the scratch words or the h
 * workspace.  This entry point computes exactly what h3fp4_swiglu_pack
 * computes (same tensor scale, QDATA and SFA bytes) with its scratch in a
 * static device array owned by the library: 256 bytes of counters plus room
 * for H3FP4_NOALLOC_MAX_ELEMENTS bf16 values of h (8 MiB in all), held by
 * every GPU that loads the library until the process exits.  It calls no
 * cudaMalloc, cudaFree or allocating library routine.
 *
 *   Arguments as for h3fp4_swiglu_pack, without scratch and h_workspace.
 *   m * f must not exceed H3FP4_NOALLOC_MAX_ELEMENTS (else H3FP4_ERR_SHAPE,
 *   nothing enqueued).
 *
 * The first call on a device looks up the array's device address (with that
 * device current) and may load the library's device code; make that first
 * call before any stream capture.  The address is kept for the life of the
 * process's context on that device: after cudaDeviceReset, do not call this
 * entry point again in that process.  All calls share the array and it keeps the
 * last call's contents (each call clears its counters and rewrites h before
 * reading it); calls whose GPU work overlaps race on it and must be
 * serialised by the caller.
 */
#define H3FP4_NOALLOC_MAX_ELEMENTS (1 << 22)
H3FP4_API h3fp4_status h3fp4_swiglu_pack_noalloc(const void *gate_bf16, int64_t ldg, const void *up_bf16,
                                                 int64_t ldu, int64_t m, int64_t m_pad, int64_t f,
                                                 float *tensor_scale, uint8_t *qdata, uint8_t *sfa,
                                                 void *stream);

/*
 * h3fp4_device_error -- reads and clears the device-side error word of the
 * current device (synchronous).  Kernels whose pipeline waits give up after
 * their time limit (2 s) record a nonzero code there instead of hanging, and
 * return.  Bits: GEMM waits 1 (a free stage), 2 (operands landed), 4 (a
 * finished accumulator), 8 (a drained accumulator), 16 (scale atoms landed);
 * 256 the cooperative producer's grid barrier.
 * Returns H3FP4_OK and stores the word in *code (0 = no error).
 */
H3FP4_API h3fp4_status h3fp4_device_error(uint32_t *code);

/*
 * Failure detection -- diagnostics, not part of the hot path.  No counterpart
 * on the source pages beyond the bounded waits themselves ("NVFP4 Streaming
 * Design", P2: a cooperative producer around a grid barrier with a bounded
 * wait).  Each call runs one of the library's kernels with a wait that cannot
 * be satisfied and a limit of limit_us microseconds (1 .. 2,000,000, else
 * H3FP4_ERR_SHAPE), so that a caller can check that a wait which runs out
 * ends the kernel with an error code instead of a hang, and that the device
 * stays usable afterwards.
 *
 * h3fp4_diag_producer_barrier_timeout -- the cooperative plain producer
 * (h3fp4_quantize_pack's kernel, same arguments and checks) with its grid
 * barrier's arrival target one above the grid size: every CTA gives up after
 * limit_us, records bit 256 and returns.  tensor_scale, qdata and sfa are not
 * written; pass 1 reads x.
 *
 * h3fp4_diag_gemm_wait_timeout -- the default GEMM kernel (same arguments
 * and checks as h3fp4_gemm, default configuration) with its operand loads
 * withheld: the scale-copy, MMA and epilogue warps' waits run out after
 * limit_us and record bits 16, 2 and 4.  c_bf16 is not written and no
 * operand is read.
 */
H3FP4_API h3fp4_status h3fp4_diag_producer_barrier_timeout(const void *x_bf16, int64_t ldx, int64_t m,
                                                           int64_t m_pad, int64_t d, float *tensor_scale,
                                                           uint32_t *scratch, uint8_t *qdata, uint8_t *sfa,
                                                           uint32_t limit_us, void *stream);
H3FP4_API h3fp4_status h3fp4_diag_gemm_wait_timeout(const uint8_t *a_q, const uint8_t *a_sf,
                                                    const float *a_tensor_scale, const uint8_t *b_q,
                                                    const uint8_t *b_sf, const float *b_tensor_scale, void *c_bf16,
                                                    int64_t ldc, int64_t m, int64_t m_pad, int64_t n, int64_t k,
                                                    uint32_t limit_us, void *stream);

/* Human-readable name of a status code (static string). */
H3FP4_API const char *h3fp4_status_string(h3fp4_status status);

/* Build description: version, target architecture, compiler. (static string) */
H3FP4_API const char *h3fp4_build_info(void);

#ifdef __cplusplus
}
#endif

#endif /* H3FP4_H */
