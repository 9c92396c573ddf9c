// gemm.cu -- block-scaled NVFP4 GEMM with the alpha epilogue, sm_103a tcgen05.
//
// C[i, j] = RN_bf16(RN_f32(ts_a * ts_b) * sum_k e2m1(a) e4m3(sfa) e2m1(b) e4m3(sfb))
// ("NVFP4 Streaming Design", Available Foundation and P0: E2M1 A/B, E4M3
// scales, FP32 accumulation, alpha applied before the BF16 conversion; "FC2
// NVFP4 Library Scheduling", Exact Operation: activation [M,K] times weight
// [N,K], both K-major, row-major BF16 output, logical rows only).
//
// Persistent kernel, one CTA per SM, 10 warps:
//   warp 0      TMA producer: per 256-wide K step, one 2-D tensor copy each for
//               the A tile (128 rows x 128 bytes) and the B tile (256 x 128 bytes),
//               both with 128-byte swizzle, plus 1-D bulk copies of the scale
//               atoms (A: 4 atoms = 2 KB, B: 2 x 2 KB), into a 4-stage ring;
//   warp 1      allocates TMEM, then one lane copies the scale atoms into TMEM
//               (tcgen05.cp 32x128b.warpx4) and issues four
//               tcgen05.mma kind::mxf4nvf4 (K = 64 each) per stage into the
//               FP32 accumulator (TMEM columns 0-255); tcgen05.commit frees the
//               stage and, after a tile's last stage, hands the accumulator to
//               the epilogue;
//   warps 2-9   epilogue: each warp drains one 32-lane quarter x 128 columns of
//               the accumulator into registers (tcgen05.ld), releases the
//               accumulator at once so that the next tile's MMAs can start, and
//               then applies alpha, converts to bf16 and stores.
// Tiles (128 x 256 outputs) are visited in groups of n_group N-tiles x all
// M-tiles with N fastest, so every 128-row A tile is used by n_group
// consecutive tiles while it is L2-resident, and the B tiles of a group stay
// resident while the group sweeps M (the N-group A-tile reuse factor).
// The scale copies of stage s live in their own 48 TMEM columns (256 + 48 s),
// so a later stage never overwrites scales an in-flight MMA still reads.
// Every pipeline wait gives up after 2 s and records a device error instead of
// hanging.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "launch.h"
#include "ptx.cuh"

namespace h3fp4 {

__device__ uint32_t g_device_error;

namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 256;             // K elements per pipeline stage
constexpr int BKB = BK / 2;         // bytes of one row per stage
constexpr int kStages = 4;
constexpr uint32_t A_BYTES = BM * BKB;   // 16 KB
constexpr uint32_t B_BYTES = BN * BKB;   // 32 KB
constexpr uint32_t ATOM = 512;           // 128 rows x 4 scales
constexpr uint32_t SFA_BYTES = 4 * ATOM; // 128 rows x 16 scales
constexpr uint32_t SFB_BYTES = 8 * ATOM; // 256 rows x 16 scales
constexpr int kEpiWarps = 8;
constexpr int kThreads = 32 * (2 + kEpiWarps);
constexpr int kDefaultNGroup = 16;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t ACC_COL = 0;
constexpr uint32_t SF_COL = 256;
constexpr uint32_t SF_COLS_PER_STAGE = 48;  // 16 for A, 32 for B
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// Device error codes (OR-ed into g_device_error).
constexpr uint32_t ERR_WAIT_EMPTY = 1u;
constexpr uint32_t ERR_WAIT_FULL = 2u;
constexpr uint32_t ERR_WAIT_ACC = 4u;
constexpr uint32_t ERR_WAIT_ACC_EMPTY = 8u;

struct __align__(1024) Smem {
    uint8_t a[kStages][A_BYTES];
    uint8_t b[kStages][B_BYTES];
    uint8_t sfa[kStages][SFA_BYTES];
    uint8_t sfb[kStages][SFB_BYTES];
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t acc_full;
    uint64_t acc_empty;
    uint32_t tmem_base;
};
constexpr size_t kSmemBytes = sizeof(Smem) + 1024;  // + slack for 1024-byte alignment

// Instruction descriptor for kind::mxf4nvf4: A and B E2M1 (format 1), both
// K-major, UE4M3 scales (bit 23 = 0), scale-factor ids 0, N >> 3 at bit 17,
// M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_nvf4(int m, int n)
{
    return (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
}

__device__ __forceinline__ void record_error(uint32_t code) { atomicOr(&g_device_error, code); }

// Output tile t of the persistent schedule: groups of n_group N-tiles x all
// M-tiles, N fastest inside a group (the last group may be narrower).
__device__ __forceinline__ void tile_coords(int t, int m_tiles, int n_tiles, int n_group, int &mt, int &nt)
{
    const int group_tiles = n_group * m_tiles;
    const int g = t / group_tiles;
    const int tt = t - g * group_tiles;
    const int ng = min(n_group, n_tiles - g * n_group);
    nt = g * n_group + tt % ng;
    mt = tt / ng;
}

__global__ void __launch_bounds__(kThreads, 1)
    nvf4_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const uint8_t *__restrict__ a_sf, const uint8_t *__restrict__ b_sf,
                     const float *__restrict__ a_ts, const float *__restrict__ b_ts, uint16_t *__restrict__ C,
                     int64_t ldc, int m, int n, int k, int m_tiles, int n_tiles, int n_group)
{
    extern __shared__ uint8_t smem_raw[];
    Smem &sm = *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int kt_count = k / BK;
    const int64_t atoms_per_rb = k / 64;           // scale atoms per 128-row block
    const int n_rb = (n + 127) / 128;
    const int total_tiles = m_tiles * n_tiles;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&sm.full[s]), 1);
            mbar_init(smem_u32(&sm.empty[s]), 1);
        }
        mbar_init(smem_u32(&sm.acc_full), 1);
        mbar_init(smem_u32(&sm.acc_empty), kEpiWarps);
        fence_mbar_init();
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&sm.tmem_base), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;

    if (warp == 0) {
        if (lane == 0) {
            uint32_t it = 0;  // global K-step counter across this CTA's tiles
            bool ok = true;
            for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
                int mt, nt;
                tile_coords(t, m_tiles, n_tiles, n_group, mt, nt);
                const bool has_rb1 = (2 * nt + 1) < n_rb;   // second 128-row half of the B tile exists
                const uint32_t tx = A_BYTES + B_BYTES + SFA_BYTES + (has_rb1 ? SFB_BYTES : SFB_BYTES / 2);
                for (int kt = 0; kt < kt_count; ++kt, ++it) {
                    const int s = it % kStages;
                    const uint32_t ph = (it / kStages) & 1;
                    if (!mbar_wait_bounded(smem_u32(&sm.empty[s]), ph ^ 1u, kWaitLimitNs)) {
                        record_error(ERR_WAIT_EMPTY);
                        ok = false;
                        break;
                    }
                    const uint32_t bar = smem_u32(&sm.full[s]);
                    mbar_arrive_expect_tx(bar, tx);
                    tma_load_2d(smem_u32(sm.a[s]), &tmA, kt * BKB, mt * BM, bar);
                    tma_load_2d(smem_u32(sm.b[s]), &tmB, kt * BKB, nt * BN, bar);
                    bulk_load(smem_u32(sm.sfa[s]), a_sf + (mt * atoms_per_rb + kt * 4) * ATOM, SFA_BYTES, bar);
                    bulk_load(smem_u32(sm.sfb[s]), b_sf + ((2 * nt) * atoms_per_rb + kt * 4) * ATOM, SFB_BYTES / 2,
                              bar);
                    if (has_rb1)
                        bulk_load(smem_u32(sm.sfb[s]) + SFB_BYTES / 2,
                                  b_sf + ((2 * nt + 1) * atoms_per_rb + kt * 4) * ATOM, SFB_BYTES / 2, bar);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_nvf4(BM, BN);
            uint32_t it = 0, local = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x, ++local) {
                // the epilogue must have drained the previous tile's accumulator
                if (!mbar_wait_bounded(smem_u32(&sm.acc_empty), (local & 1) ^ 1u, kWaitLimitNs)) {
                    record_error(ERR_WAIT_ACC_EMPTY);
                    break;
                }
                tc_fence_after();
                for (int kt = 0; kt < kt_count; ++kt, ++it) {
                    const int s = it % kStages;
                    const uint32_t ph = (it / kStages) & 1;
                    if (!mbar_wait_bounded(smem_u32(&sm.full[s]), ph, kWaitLimitNs)) {
                        record_error(ERR_WAIT_FULL);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sfa_t = tmem + SF_COL + s * SF_COLS_PER_STAGE;
                    const uint32_t sfb_t = sfa_t + 16;
                    const uint32_t sfa_s = smem_u32(sm.sfa[s]);
                    const uint32_t sfb_s = smem_u32(sm.sfb[s]);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        tc_cp_32x128b_warpx4(sfa_t + 4 * j, smem_desc(sfa_s + j * ATOM, 0, 128, 0));
                        tc_cp_32x128b_warpx4(sfb_t + 8 * j, smem_desc(sfb_s + j * ATOM, 0, 128, 0));
                        tc_cp_32x128b_warpx4(sfb_t + 8 * j + 4,
                                             smem_desc(sfb_s + SFB_BYTES / 2 + j * ATOM, 0, 128, 0));
                    }
                    const uint64_t a_desc = smem_desc(smem_u32(sm.a[s]), 0, 1024, 2);
                    const uint64_t b_desc = smem_desc(smem_u32(sm.b[s]), 0, 1024, 2);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        // K step j: 64 elements = 32 bytes further along the swizzled row.
                        tc_mma_nvf4(tmem + ACC_COL, a_desc + 2 * j, b_desc + 2 * j, idesc, sfa_t + 4 * j,
                                    sfb_t + 8 * j, (kt | j) != 0);
                    }
                    tc_commit(smem_u32(&sm.empty[s]));
                }
                if (ok)
                    tc_commit(smem_u32(&sm.acc_full));
            }
        }
    } else {
        const int q = warp & 3;              // TMEM lane quarter this warp may access
        const int half = (warp - 2) >> 2;    // which 128 accumulator columns it drains
        const float alpha = __fmul_rn(*a_ts, *b_ts);
        uint32_t local = 0;
        for (int t = blockIdx.x; t < total_tiles; t += gridDim.x, ++local) {
            int mt, nt;
            tile_coords(t, m_tiles, n_tiles, n_group, mt, nt);
            bool ok = false;
            if (lane == 0)
                ok = mbar_wait_bounded(smem_u32(&sm.acc_full), local & 1, kWaitLimitNs);
            ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
            __syncwarp();
            if (!ok) {
                if (lane == 0)
                    record_error(ERR_WAIT_ACC);
                break;
            }
            tc_fence_after();
            uint32_t v[4][32];
            const uint32_t base = tmem + (static_cast<uint32_t>(q * 32) << 16) + ACC_COL + half * 128;
#pragma unroll
            for (int c = 0; c < 4; ++c)
                tmem_ld_32x32b_x32(base + 32 * c, v[c]);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_u32(&sm.acc_empty));   // accumulator free for the next tile

            const int row = mt * BM + q * 32 + lane;
            const int col0 = nt * BN + half * 128;
            if (row < m && col0 < n) {
                uint4 *dst = reinterpret_cast<uint4 *>(C + static_cast<int64_t>(row) * ldc + col0);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t p[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float lo = __fmul_rn(alpha, __uint_as_float(v[c][2 * i]));
                        const float hi = __fmul_rn(alpha, __uint_as_float(v[c][2 * i + 1]));
                        const __nv_bfloat162 b2 = __floats2bfloat162_rn(lo, hi);
                        memcpy(&p[i], &b2, 4);
                    }
                    dst[4 * c + 0] = make_uint4(p[0], p[1], p[2], p[3]);
                    dst[4 * c + 1] = make_uint4(p[4], p[5], p[6], p[7]);
                    dst[4 * c + 2] = make_uint4(p[8], p[9], p[10], p[11]);
                    dst[4 * c + 3] = make_uint4(p[12], p[13], p[14], p[15]);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 2-D uint8 tensor map over a K-major packed operand [rows, k/2] with a box of
// 128 bytes x box_rows and 128-byte swizzle (rows past `rows` read as zero).
bool make_operand_map(CUtensorMap *tm, const void *base, int64_t rows, int64_t kbytes, uint32_t box_rows)
{
    auto fn = encode_fn();
    if (!fn)
        return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(kbytes), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(kbytes)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(BKB), box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace

h3fp4_status launch_gemm(const uint8_t *a_q, const uint8_t *a_sf, const float *a_ts, const uint8_t *b_q,
                         const uint8_t *b_sf, const float *b_ts, uint16_t *c, int64_t ldc, int64_t m, int64_t m_pad,
                         int64_t n, int64_t k, const h3fp4_gemm_config &cfg, cudaStream_t st)
{
    (void)cfg;
    if (m == 0 || n == 0)
        return H3FP4_OK;
    CUtensorMap tmA, tmB;
    if (!make_operand_map(&tmA, a_q, m_pad, k / 2, BM) || !make_operand_map(&tmB, b_q, n, k / 2, BN))
        return H3FP4_ERR_CUDA;
    static bool attr_set[64] = {false};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return H3FP4_ERR_CUDA;
    if (dev >= 0 && dev < 64 && !attr_set[dev]) {
        if (cudaFuncSetAttribute(nvf4_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kSmemBytes)) != cudaSuccess)
            return H3FP4_ERR_CUDA;
        attr_set[dev] = true;
    }
    const int m_tiles = static_cast<int>((m + BM - 1) / BM);
    const int n_tiles = static_cast<int>((n + BN - 1) / BN);
    const int64_t total = static_cast<int64_t>(m_tiles) * n_tiles;
    if (total > 0x7FFFFFFF)
        return H3FP4_ERR_SHAPE;
    int n_group = cfg.n_group > 0 ? cfg.n_group : kDefaultNGroup;
    if (n_group > n_tiles)
        n_group = n_tiles;
    const int grid = static_cast<int>(total < sm_count() ? total : sm_count());
    nvf4_gemm_kernel<<<grid, kThreads, kSmemBytes, st>>>(tmA, tmB, a_sf, b_sf, a_ts, b_ts, c, ldc,
                                                        static_cast<int>(m), static_cast<int>(n),
                                                        static_cast<int>(k), m_tiles, n_tiles, n_group);
    return cudaGetLastError() == cudaSuccess ? H3FP4_OK : H3FP4_ERR_CUDA;
}

h3fp4_status read_device_error(uint32_t *code)
{
    uint32_t v = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v)) != cudaSuccess)
        return H3FP4_ERR_CUDA;
    const uint32_t zero = 0;
    if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero)) != cudaSuccess)
        return H3FP4_ERR_CUDA;
    *code = v;
    return H3FP4_OK;
}

}  // namespace h3fp4
