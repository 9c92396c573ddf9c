// gemm.cu -- block-scaled NVFP4 GEMM with the alpha epilogue, sm_103a tcgen05.
//
// C[i, j] = RN_bf16(RN_f32(ts_a * ts_b) * sum_k e2m1(a) e4m3(sfa) e2m1(b) e4m3(sfb))
// ("NVFP4 Streaming Design", Available Foundation and P0: E2M1 A/B, E4M3
// scales, FP32 accumulation, alpha applied before the BF16 conversion; "FC2
// NVFP4 Library Scheduling", Exact Operation: activation [M,K] times weight
// [N,K], both K-major, row-major BF16 output, logical rows only).
//
// Two kernels behind h3fp4_gemm (h3fp4_gemm_config.cta_pair), both
// persistent, TMA-fed, with FP32 accumulators in TMEM and tcgen05.mma
// kind::mxf4nvf4 block_scale scale_vec::4X, each 256-element K stage covered
// by two K = 96 instructions and one K = 64 (see kStageMmas):
//   0 / 4 (default)  CTA pairs (cta_group::2) on 256 x 256 output tiles: per K
//                step each CTA loads its 128 rows of A and of B and the step's
//                scale atoms; in the leader, two copy warps copy the atoms into
//                TMEM with tcgen05.cp and one MMA warp issues the three pair
//                MMAs, every tcgen05 instruction issued warp-collectively
//                through elect.sync (see the paircp namespace below);
//   1            one CTA per 128 x 256 tile; four scale warps move the atoms
//                into TMEM with tcgen05.st; one lane issues the MMAs.
// Every operand load is a plain (non-multicast) TMA copy into the issuing
// CTA's own shared memory.
// Shared by both: the epilogue warps drain 32 TMEM lanes x 128 columns each
// (tcgen05.ld), apply alpha and round to bf16 as they go, release the
// accumulator at once so that the next tile's MMAs can start, and write their
// block with 16-column TMA tensor stores staged through shared memory (per-lane
// stores from the row-per-lane accumulator layout touch 32 rows per
// instruction and measured 18% slower end to end); optionally the gated
// residual epilogue.  Tiles are visited in groups of n_group N-tiles x all
// M-tiles with N fastest, so every A row block is used by n_group consecutive
// tiles while it is L2-resident and a group's B tiles stay resident while it
// sweeps M (the N-group A-tile reuse factor).  A stage's scales live in TMEM
// columns of their own, rewritten only after the MMAs that read them have
// committed.  Every pipeline wait gives up after 2 s and records a device
// error instead of hanging.
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
constexpr int kScaleWarps = 4;                     // one per TMEM lane quarter
constexpr int kFirstEpiWarp = 2;
constexpr int kFirstScaleWarp = kFirstEpiWarp + kEpiWarps;
constexpr int kThreads = 32 * (2 + kEpiWarps + kScaleWarps);
constexpr int kDefaultNGroup = 28;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t ACC_COL = 0;
constexpr uint32_t SF_COL = 256;
constexpr uint32_t SF_COLS_PER_STAGE = 48;  // 16 for A, 32 for B
constexpr int CST_COLS = 16;                // output columns per tensor store (32 rows x 32 bytes)
constexpr uint32_t CST_BYTES = 32 * CST_COLS * 2;
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// Device error codes (OR-ed into g_device_error).
constexpr uint32_t ERR_WAIT_EMPTY = 1u;
constexpr uint32_t ERR_WAIT_FULL = 2u;
constexpr uint32_t ERR_WAIT_ACC = 4u;
constexpr uint32_t ERR_WAIT_ACC_EMPTY = 8u;
constexpr uint32_t ERR_WAIT_SCALES = 16u;

struct __align__(1024) Smem {
    uint8_t a[kStages][A_BYTES];
    uint8_t b[kStages][B_BYTES];
    uint8_t sfa[kStages][SFA_BYTES];
    uint8_t sfb[kStages][SFB_BYTES];
    uint8_t cst[kEpiWarps][CST_BYTES];  // per epilogue warp: output staging for tensor stores
    uint64_t res_full[kEpiWarps];       // per epilogue warp: a residual block landed in cst (gated epilogue)
    uint64_t full[kStages];      // A and B tiles landed
    uint64_t sf_full[kStages];   // scale atoms landed
    uint64_t empty[kStages];
    uint64_t sf_ready[kStages];  // scales staged in TMEM
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

// The block-scaled MMAs of one 256-element K stage.  On sm_103a the
// instruction descriptor's bit 31 selects a dense K of 96 instead of 64 for
// the E2M1 kinds: 1.5x the work per instruction in about the same tensor-pipe
// time (a one-CTA microbenchmark: 43.6k against 28.2k FLOP per SM clock).
// One instruction may not cross the 128-byte swizzled row that holds a
// stage's 256 elements of an operand row, so a stage takes K = 96 at elements
// 0 and 96 and K = 64 at element 192: three instructions instead of four.  The
// scale-factor id (descriptor bits 29-30 for A, 4-5 for B) is the byte of the
// 32-bit TMEM scale word at which the instruction's first scale sits: the
// second K = 96 MMA starts at scale block 6, byte 2 of the word that holds
// blocks 4-7, and reads on into the next word.
constexpr int kStageMmas = 3;
__host__ __device__ constexpr uint32_t stage_mma_k0(int j) { return j == 0 ? 0u : (j == 1 ? 96u : 192u); }
// descriptor start-address advance, in 16-byte units (two E2M1 values per byte)
__host__ __device__ constexpr uint32_t stage_mma_desc(int j) { return stage_mma_k0(j) / 32; }
// the group of 4 scale blocks (one 128x4 atom, one TMEM column per 32 rows) holding the first scale
__host__ __device__ constexpr uint32_t stage_mma_chunk(int j) { return stage_mma_k0(j) / 64; }
__host__ __device__ constexpr uint32_t stage_mma_idesc(uint32_t base, int j)
{
    return j < 2 ? base | (1u << 31) | (((stage_mma_k0(j) / 16) % 4) << 29) | (((stage_mma_k0(j) / 16) % 4) << 4)
                 : base;
}
static_assert(stage_mma_k0(1) + 96 <= stage_mma_k0(2) && stage_mma_k0(2) + 64 == 256, "a stage covers K = 256");

__device__ __forceinline__ void record_error(uint32_t code) { atomicOr(&g_device_error, code); }

// Bounded wait on behalf of a whole warp; the outcome is warp-uniform.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns = kWaitLimitNs)
{
    // Every lane polls: polling from lane 0 alone and broadcasting the outcome
    // measured 4-13% slower (a later wake-up of the other lanes).
    const bool ok = mbar_wait_bounded(bar, parity, limit_ns);
    return __all_sync(0xFFFFFFFFu, ok);
}

// As warp_wait, but polling with the non-blocking test_wait instead of a
// suspending try_wait: for a warp whose wake-up latency sits on the critical
// path (the default GEMM's MMA warp: 1.2 % faster), at the price of issue
// slots while it spins.  Bounded like every other wait.
__device__ __forceinline__ bool warp_wait_spin(uint32_t bar, uint32_t parity, uint64_t limit_ns = kWaitLimitNs)
{
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (__all_sync(0xFFFFFFFFu, mbar_test_wait(bar, parity)))
            return true;
        if (globaltimer_ns() - t0 > limit_ns)
            return false;
    }
}

// The scale layout the block-scaled MMA reads from TMEM: for MMA K step j,
// row i (16 bytes) of the 128x4 atom goes to columns 4j .. 4j+3 of lane
// 32q + i for every lane quarter q, i.e. the layout of a tcgen05.cp
// .32x128b.warpx4 copy of the atom.  SFA (4 atoms, one per K step) takes 16
// columns; SFB (two 128-row halves x 4 atoms) takes 32 columns, step j and
// half h at 8j + 4h.  read_scales gathers, for one lane, the words it writes:
// a[] for SFA, b[] for SFB.
__device__ __forceinline__ void read_scales(const uint8_t *sfa, const uint8_t *sfb, int lane, uint32_t (&a)[16],
                                            uint32_t (&b)[32])
{
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint4 v = *reinterpret_cast<const uint4 *>(sfa + j * ATOM + lane * 16);
        a[4 * j + 0] = v.x;
        a[4 * j + 1] = v.y;
        a[4 * j + 2] = v.z;
        a[4 * j + 3] = v.w;
    }
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint4 v = *reinterpret_cast<const uint4 *>(sfb + h * (4 * ATOM) + j * ATOM + lane * 16);
            b[8 * j + 4 * h + 0] = v.x;
            b[8 * j + 4 * h + 1] = v.y;
            b[8 * j + 4 * h + 2] = v.z;
            b[8 * j + 4 * h + 3] = v.w;
        }
}

// Moves one stage's scale atoms from shared memory into TMEM (SFA at sfa_col,
// SFB at sfb_col).  Executed by a whole warp; `lane_base` selects the warp's
// lane quarter.  One tcgen05.st per operand replaces twelve tcgen05.cp in the
// tensor pipe.
__device__ __forceinline__ void stage_scales(uint32_t lane_base, uint32_t sfa_col, uint32_t sfb_col,
                                             const uint8_t *sfa, const uint8_t *sfb, int lane)
{
    uint32_t a[16], b[32];
    read_scales(sfa, sfb, lane, a, b);
    tmem_st_32x32b_x16(lane_base + sfa_col, a);
    tmem_st_32x32b_x32(lane_base + sfb_col, b);
    tmem_st_wait();
}

// Writes one epilogue warp's 32 output rows x 128 bf16 columns (row = lane;
// pk[i] holds columns 2i and 2i+1) with 16-column tensor stores through the
// warp's 1 KB shared-memory buffer.  The per-lane global stores this replaces
// wrote 16 bytes into each of 32 different rows per instruction; a tensor
// store moves whole 32-byte row pieces of the 32 x 16 block.  Rows at or past
// the tensor map's M extent (the padding of the last M tile) are not written.
__device__ __forceinline__ void store_rows(const CUtensorMap *tmC, uint32_t buf, const uint32_t (&pk)[64], int col0,
                                          int row0, int lane)
{
#pragma unroll
    for (int c = 0; c < 128 / CST_COLS; ++c) {
        if (lane == 0)
            bulk_wait_group_read0();   // the previous store has finished reading the buffer
        __syncwarp();
        const int w = c * (CST_COLS / 2);
        st_shared_v4(buf + lane * 32, pk[w], pk[w + 1], pk[w + 2], pk[w + 3]);
        st_shared_v4(buf + lane * 32 + 16, pk[w + 4], pk[w + 5], pk[w + 6], pk[w + 7]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            tma_store_2d(tmC, buf, col0 + c * CST_COLS, row0);
            bulk_commit_group();
        }
    }
}

// Arguments of the gated residual epilogue: gate [nseg, n] bf16 (leading
// dimension ld_gate) selected per output row by the row segments off[0..nseg].
struct GatedEpilogue {
    const uint16_t *gate;
    int64_t ld_gate;
    int32_t off[H3FP4_MAX_SEGMENTS + 1];
    int32_t nseg;
};

// Segment of row r: the number of interior boundaries off[1..nseg-1] at or
// below r (fully unrolled, constant indices, so the table stays in
// kernel-parameter space).
__device__ __forceinline__ const uint16_t *gate_row(const GatedEpilogue &ge, int r)
{
    int s = 0;
#pragma unroll
    for (int i = 1; i < H3FP4_MAX_SEGMENTS; ++i)
        s += (i < ge.nseg && r >= ge.off[i]) ? 1 : 0;
    return ge.gate + static_cast<int64_t>(s) * ge.ld_gate;
}

__device__ __forceinline__ uint32_t bf2_mul_rn(uint32_t a, uint32_t b)
{
    __nv_bfloat162 x, y;
    memcpy(&x, &a, 4);
    memcpy(&y, &b, 4);
    const __nv_bfloat162 r = __hmul2_rn(x, y);
    uint32_t u;
    memcpy(&u, &r, 4);
    return u;
}

__device__ __forceinline__ uint32_t bf2_add_rn(uint32_t a, uint32_t b)
{
    __nv_bfloat162 x, y;
    memcpy(&x, &a, 4);
    memcpy(&y, &b, 4);
    const __nv_bfloat162 r = __hadd2_rn(x, y);
    uint32_t u;
    memcpy(&u, &r, 4);
    return u;
}

// Gated residual form of store_rows ("NVFP4 Streaming Design", P4: the
// explicit BF16 conversion, gate multiply, residual add and final BF16
// rounding): out = RN_bf16(res + RN_bf16(gate * c)) with c the BF16 GEMM
// result held in pk.  Per 16-column block the warp loads its 32 x 16
// residual block into its buffer with a tensor copy (rows past the tensor
// map's M extent read as zero), combines it in registers with correctly
// rounded bf16x2 multiply and add, writes the result back into the buffer and
// stores it with a tensor store.  `res` may be the output itself: each block
// is read before it is written, by the same warp.
__device__ __forceinline__ bool store_rows_gated(const CUtensorMap *tmC, const CUtensorMap *tmR, uint32_t buf,
                                                 uint32_t bar, uint32_t &phase, const uint32_t (&pk)[64], int col0,
                                                 int row0, int lane, const uint16_t *grow)
{
#pragma unroll   // constant indices into pk keep it in registers
    for (int c = 0; c < 128 / CST_COLS; ++c) {
        if (lane == 0) {
            bulk_wait_group_read0();   // the previous store has finished reading the buffer
            mbar_arrive_expect_tx(bar, CST_BYTES);
            tma_load_2d(buf, tmR, col0 + c * CST_COLS, row0, bar);
        }
        __syncwarp();
        // every lane waits on the barrier (the residual block written by the copy engine)
        if (!warp_wait(bar, phase))
            return false;
        phase ^= 1u;
        const uint4 r0 = ld_shared_v4(buf + lane * 32);
        const uint4 r1 = ld_shared_v4(buf + lane * 32 + 16);
        const uint4 g0 = *reinterpret_cast<const uint4 *>(grow + col0 + c * CST_COLS);
        const uint4 g1 = *reinterpret_cast<const uint4 *>(grow + col0 + c * CST_COLS + 8);
        const uint32_t rw[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
        const uint32_t gw[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
        uint32_t o[8];
        const int w = c * (CST_COLS / 2);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            o[i] = bf2_add_rn(rw[i], bf2_mul_rn(gw[i], pk[w + i]));
        __syncwarp();   // every lane has read the residual before any lane overwrites the buffer
        st_shared_v4(buf + lane * 32, o[0], o[1], o[2], o[3]);
        st_shared_v4(buf + lane * 32 + 16, o[4], o[5], o[6], o[7]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            tma_store_2d(tmC, buf, col0 + c * CST_COLS, row0);
            bulk_commit_group();
        }
    }
    return true;
}

// store_rows_gated with the residual blocks prefetched through a ring of NB
// 1 KB buffers (NB - 1 loads ahead), so that their load latency overlaps the
// blocks being combined and stored instead of being paid once per block.
// bars are NB mbarriers 8 bytes apart; bit b of `phases` is buffer b's phase.
// A buffer is reloaded only after every earlier store of the warp has
// finished reading shared memory (the last user of the buffer is the store of
// the block NB - 1 places back).
template <int NB>
__device__ __forceinline__ bool store_rows_gated_ring(const CUtensorMap *tmC, const CUtensorMap *tmR, uint32_t buf,
                                                      uint32_t bars, uint32_t &phases, const uint32_t (&pk)[64],
                                                      int col0, int row0, int lane, const uint16_t *grow)
{
    constexpr int NC = 128 / CST_COLS;
    if (lane == 0) {
        bulk_wait_group_read0();   // the previous tile's stores have finished reading the buffers
#pragma unroll
        for (int c = 0; c < NB - 1; ++c) {
            mbar_arrive_expect_tx(bars + 8 * c, CST_BYTES);
            tma_load_2d(buf + c * CST_BYTES, tmR, col0 + c * CST_COLS, row0, bars + 8 * c);
        }
    }
#pragma unroll   // constant indices into pk keep it in registers
    for (int c = 0; c < NC; ++c) {
        const int b = c % NB;
        if (c + NB - 1 < NC && lane == 0) {
            const int bp = (c + NB - 1) % NB;
            bulk_wait_group_read0();   // block c - 1's store, the last reader of buffer bp, is done with it
            mbar_arrive_expect_tx(bars + 8 * bp, CST_BYTES);
            tma_load_2d(buf + bp * CST_BYTES, tmR, col0 + (c + NB - 1) * CST_COLS, row0, bars + 8 * bp);
        }
        __syncwarp();
        if (!warp_wait(bars + 8 * b, (phases >> b) & 1u))
            return false;
        phases ^= 1u << b;
        const uint32_t bb = buf + b * CST_BYTES;
        const uint4 r0 = ld_shared_v4(bb + lane * 32);
        const uint4 r1 = ld_shared_v4(bb + lane * 32 + 16);
        const uint4 g0 = *reinterpret_cast<const uint4 *>(grow + col0 + c * CST_COLS);
        const uint4 g1 = *reinterpret_cast<const uint4 *>(grow + col0 + c * CST_COLS + 8);
        const uint32_t rw[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
        const uint32_t gw[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
        uint32_t o[8];
        const int w = c * (CST_COLS / 2);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            o[i] = bf2_add_rn(rw[i], bf2_mul_rn(gw[i], pk[w + i]));
        __syncwarp();   // every lane has read the residual before any lane overwrites the buffer
        st_shared_v4(bb + lane * 32, o[0], o[1], o[2], o[3]);
        st_shared_v4(bb + lane * 32 + 16, o[4], o[5], o[6], o[7]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            tma_store_2d(tmC, bb, col0 + c * CST_COLS, row0);
            bulk_commit_group();
        }
    }
    return true;
}

// Output tile t of the persistent schedule: groups of n_group N-tiles x all
// M-tiles, N fastest inside a group (the last group may be narrower).  Odd
// groups sweep M backwards, so that a group starts on the A row blocks the
// previous one read last, still partly in L2 (full QKV: DRAM reads 607 ->
// 592 MB per launch, same time).
__device__ __forceinline__ void tile_coords(int t, int m_tiles, int n_tiles, int n_group, int &mt, int &nt)
{
    const int group_tiles = n_group * m_tiles;
    const int g = t / group_tiles;
    const int tt = t - g * group_tiles;
    const int ng = min(n_group, n_tiles - g * n_group);
    nt = g * n_group + tt % ng;
    mt = tt / ng;
    if (g & 1)
        mt = m_tiles - 1 - mt;
}

// One CTA per 128 x 256 output tile: warp 0 loads A, B and their scale atoms
// into a 4-stage ring, four scale warps move each stage's atoms into TMEM with
// tcgen05.st, one lane of warp 1 issues the MMAs, eight warps drain the
// accumulator.
template <bool kGated>
__global__ void __launch_bounds__(kThreads, 1)
    nvf4_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmR,
                     const __grid_constant__ GatedEpilogue ge, const uint8_t *__restrict__ a_sf,
                     const uint8_t *__restrict__ b_sf, const float *__restrict__ a_ts,
                     const float *__restrict__ b_ts, int m, int n, int k, int m_tiles, int n_tiles, int n_group)
{
    extern __shared__ uint8_t smem_raw[];
    Smem &sm = *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int kt_count = k / BK;
    const int64_t atoms_per_rb = k / 64;           // scale atoms per 128-row block
    const int n_rb = (n + 127) / 128;
    const int sched_first = static_cast<int>(blockIdx.x);
    const int sched_step = static_cast<int>(gridDim.x);
    const int total_tiles = m_tiles * n_tiles;
    auto coords = [&](int t, int &mt, int &nt) { tile_coords(t, m_tiles, n_tiles, n_group, mt, nt); };

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&sm.full[s]), 1);
            mbar_init(smem_u32(&sm.sf_full[s]), 1);
            mbar_init(smem_u32(&sm.empty[s]), 1);
            mbar_init(smem_u32(&sm.sf_ready[s]), kScaleWarps);
        }
        mbar_init(smem_u32(&sm.acc_full), 1);
        mbar_init(smem_u32(&sm.acc_empty), kEpiWarps);
        for (int w = 0; w < kEpiWarps; ++w)
            mbar_init(smem_u32(&sm.res_full[w]), 1);
        fence_mbar_init();
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
        prefetch_tmap(&tmC);
        if (kGated)
            prefetch_tmap(&tmR);
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
            for (int t = sched_first; t < total_tiles && ok; t += sched_step) {
                int mt, nt;
                coords(t, mt, nt);
                const bool has_rb1 = (2 * nt + 1) < n_rb;   // second 128-row half of the B tile exists
                const uint32_t sf_tx = SFA_BYTES + (has_rb1 ? SFB_BYTES : SFB_BYTES / 2);
                for (int kt = 0; kt < kt_count; ++kt, ++it) {
                    const int s = it % kStages;
                    const uint32_t ph = (it / kStages) & 1;
                    if (!mbar_wait_bounded(smem_u32(&sm.empty[s]), ph ^ 1u, kWaitLimitNs)) {
                        record_error(ERR_WAIT_EMPTY);
                        ok = false;
                        break;
                    }
                    // scales first (small; the scale warps stage them while A and B are in flight)
                    const uint32_t sbar = smem_u32(&sm.sf_full[s]);
                    mbar_arrive_expect_tx(sbar, sf_tx);
                    bulk_load(smem_u32(sm.sfa[s]), a_sf + (mt * atoms_per_rb + kt * 4) * ATOM, SFA_BYTES, sbar);
                    bulk_load(smem_u32(sm.sfb[s]), b_sf + ((2 * nt) * atoms_per_rb + kt * 4) * ATOM, SFB_BYTES / 2,
                              sbar);
                    if (has_rb1)
                        bulk_load(smem_u32(sm.sfb[s]) + SFB_BYTES / 2,
                                  b_sf + ((2 * nt + 1) * atoms_per_rb + kt * 4) * ATOM, SFB_BYTES / 2, sbar);
                    const uint32_t bar = smem_u32(&sm.full[s]);
                    mbar_arrive_expect_tx(bar, A_BYTES + B_BYTES);
                    tma_load_2d(smem_u32(sm.a[s]), &tmA, kt * BKB, mt * BM, bar);
                    tma_load_2d(smem_u32(sm.b[s]), &tmB, kt * BKB, nt * BN, bar);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_nvf4(BM, BN);
            uint32_t it = 0, local = 0;
            bool ok = true;
            for (int t = sched_first; t < total_tiles && ok; t += sched_step, ++local) {
                // the epilogue must have drained the previous tile's accumulator
                if (!mbar_wait_bounded(smem_u32(&sm.acc_empty), (local & 1) ^ 1u, kWaitLimitNs)) {
                    record_error(ERR_WAIT_ACC_EMPTY);
                    break;
                }
                tc_fence_after();
                for (int kt = 0; kt < kt_count; ++kt, ++it) {
                    const int s = it % kStages;
                    const uint32_t ph = (it / kStages) & 1;
                    // A and B landed, and the scale warps have put this stage's scales in TMEM
                    if (!mbar_wait_bounded(smem_u32(&sm.full[s]), ph, kWaitLimitNs) ||
                        !mbar_wait_bounded(smem_u32(&sm.sf_ready[s]), ph, kWaitLimitNs)) {
                        record_error(ERR_WAIT_FULL);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sfa_t = tmem + SF_COL + s * SF_COLS_PER_STAGE;
                    const uint32_t sfb_t = sfa_t + 16;
                    const uint64_t a_desc = smem_desc(smem_u32(sm.a[s]), 0, 1024, 2);
                    const uint64_t b_desc = smem_desc(smem_u32(sm.b[s]), 0, 1024, 2);
#pragma unroll
                    for (int j = 0; j < kStageMmas; ++j)
                        tc_mma_nvf4(tmem + ACC_COL, a_desc + stage_mma_desc(j), b_desc + stage_mma_desc(j),
                                    stage_mma_idesc(idesc, j), sfa_t + 4 * stage_mma_chunk(j),
                                    sfb_t + 8 * stage_mma_chunk(j), (kt | j) != 0);
                    tc_commit(smem_u32(&sm.empty[s]));
                }
                if (ok)
                    tc_commit(smem_u32(&sm.acc_full));
            }
        }
    } else if (warp >= kFirstScaleWarp) {
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
        uint32_t it = 0;
        for (int t = sched_first; t < total_tiles; t += sched_step) {
            bool ok = true;
            for (int kt = 0; kt < kt_count; ++kt, ++it) {
                const int s = it % kStages;
                const uint32_t ph = (it / kStages) & 1;
                if (!warp_wait(smem_u32(&sm.sf_full[s]), ph)) {
                    if (lane == 0)
                        record_error(ERR_WAIT_SCALES);
                    ok = false;
                    break;
                }
                stage_scales(tmem + lane_base, SF_COL + s * SF_COLS_PER_STAGE, SF_COL + s * SF_COLS_PER_STAGE + 16,
                             sm.sfa[s], sm.sfb[s], lane);
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(smem_u32(&sm.sf_ready[s]));
            }
            if (!ok)
                break;
        }
    } else {
        const int q = warp & 3;                          // TMEM lane quarter this warp may access
        const int half = (warp - kFirstEpiWarp) >> 2;    // which 128 accumulator columns it drains
        const float alpha = __fmul_rn(*a_ts, *b_ts);
        uint32_t local = 0, rphase = 0;
        for (int t = sched_first; t < total_tiles; t += sched_step, ++local) {
            int mt, nt;
            coords(t, mt, nt);
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
            // Drain 32 columns at a time, applying alpha and rounding to bf16 at
            // once, so that only the packed half-width results stay live.
            uint32_t pk[64];
            const uint32_t base = tmem + (static_cast<uint32_t>(q * 32) << 16) + ACC_COL + half * 128;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t v[32];
                tmem_ld_32x32b_x32(base + 32 * c, v);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float lo = __fmul_rn(alpha, __uint_as_float(v[2 * i]));
                    const float hi = __fmul_rn(alpha, __uint_as_float(v[2 * i + 1]));
                    const __nv_bfloat162 b2 = __floats2bfloat162_rn(lo, hi);
                    memcpy(&pk[16 * c + i], &b2, 4);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_u32(&sm.acc_empty));   // accumulator free for the next tile
            if (kGated) {
                const int row0 = mt * BM + q * 32;
                if (!store_rows_gated(&tmC, &tmR, smem_u32(sm.cst[warp - kFirstEpiWarp]),
                                      smem_u32(&sm.res_full[warp - kFirstEpiWarp]), rphase, pk, nt * BN + half * 128,
                                      row0, lane, gate_row(ge, row0 + lane))) {
                    if (lane == 0)
                        record_error(ERR_WAIT_ACC);
                    break;
                }
            } else {
                store_rows(&tmC, smem_u32(sm.cst[warp - kFirstEpiWarp]), pk, nt * BN + half * 128, mt * BM + q * 32,
                           lane);
            }
        }
        if (lane == 0)
            bulk_wait_group0();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ---------------------------------------------------------------------------
// CTA-pair kernel with the scales copied into TMEM by tcgen05.cp
// (cta_group::2).  Per K step each CTA loads, into one stage of a 5-stage
// ring, its A scale atoms and all 256 rows' B scale atoms (onto the leader's
// sf_full barrier), then its 128 rows of A and 128 rows of B (onto the
// leader's full barrier) -- the cta_group::2 form of the tensor copy;
// out-of-range boxes, e.g. the absent second row block of the last M tile,
// are zero-filled and still count their full size.  In the leader, two copy
// warps wait for a stage's scales and copy its 12 atoms (6 each) into both
// CTAs' TMEM slot for the stage (each CTA's shared memory into its own TMEM),
// each committing to the same full barrier, which therefore completes once
// A and B have landed and the scales are in TMEM (3 arrivals: the producer's
// expect-tx and the two commits); the MMA warp waits for it, issues the
// stage's three pair MMAs (K = 96, 96, 64) and commits the stage free in both
// CTAs.  These
// warps run their loops warp-collectively, each tcgen05 instruction issued by
// one elected lane.  What the tensor pipe waits on is the issuing warps'
// per-stage time (a satisfied barrier wait alone costs ~100 cycles, a tcgen05
// instruction ~30): one warp issuing 12 copies and 4 MMAs per stage kept the
// pipe ~65 % busy; with the copies in two warps of their own, overlapping the
// A/B loads, the same GEMM runs 12 % faster.  No scale warps and no per-step
// hand-off between the SMs other than the loads' own completion.  Each CTA's
// epilogue drains its own 128 accumulator rows; kGated selects the gated
// residual epilogue.
// ---------------------------------------------------------------------------
namespace paircp {

constexpr int PBM = 128;                         // rows per CTA; the pair covers 256
constexpr int PBN = 256;                         // output columns per pair tile
constexpr uint32_t SF_ROW = 256;                 // row length of the scale tensor maps
constexpr int kFirstCopyWarp = 2;                   // leader: warps 2 and 3 copy the scale atoms into TMEM
constexpr int kCopyWarps = 2;
constexpr int kFirstEpi = kFirstCopyWarp + kCopyWarps;   // epilogue warps 4 .. 11
constexpr int kThreadsPair = 32 * (kFirstEpi + kEpiWarps);
constexpr int kResBufs = 4;                         // gated epilogue: residual blocks in flight per warp

// Stage geometry: BK = 256 K-elements per stage (128-byte operand rows with the
// 128-byte swizzle), 5 stages.  (Stages of K = 128 -- 64-byte rows, 10 stages,
// the same bytes in flight -- measured 35-50 % slower: the per-stage waits and
// commits double, and the issuing warps' per-stage costs are what the pipe
// waits on.)
struct Geo {
    static constexpr int kStages = 5;
    static constexpr int kChunks = BK / 64;                 // scale atoms (4 scale blocks each) per 128 rows
    static constexpr uint32_t ROW = BKB;                    // bytes of one operand row per stage
    static constexpr uint32_t A_BYTES = 128 * ROW;          // this CTA's 128 rows of A
    static constexpr uint32_t B_BYTES = 128 * ROW;          // this CTA's 128 rows of B
    static constexpr uint32_t SFA_BYTES = kChunks * ATOM;     // this CTA's A scale atoms
    static constexpr uint32_t SFB_BYTES = 2 * kChunks * ATOM; // all 256 B rows' scale atoms
    static constexpr uint32_t AB_TX = 2 * (A_BYTES + B_BYTES);        // both CTAs' operands of a stage
    static constexpr uint32_t SF_TX = 2 * (SFA_BYTES + SFB_BYTES);    // both CTAs' scale atoms of a stage
    static constexpr uint32_t SF_COLS = 12 * kChunks;       // TMEM columns of one stage's scales
    static constexpr uint32_t LAYOUT = 2;                   // descriptor swizzle mode: 128 B
    static constexpr uint32_t SBO = 8 * ROW;                // bytes between 8-row core-matrix groups
    static_assert(SF_COL + kStages * SF_COLS <= TMEM_COLS, "TMEM scale slots");
};

struct __align__(1024) Smem {
    using G = Geo;
    uint8_t a[G::kStages][G::A_BYTES];
    uint8_t b[G::kStages][G::B_BYTES];
    uint8_t sfa[G::kStages][G::SFA_BYTES];
    uint8_t sfb[G::kStages][G::SFB_BYTES];
    uint8_t cst[kEpiWarps][kResBufs][CST_BYTES];   // per epilogue warp: staging for tensor loads and stores
    uint64_t res_full[kEpiWarps][kResBufs];        // per epilogue warp and buffer: a residual block landed
    uint64_t full[G::kStages];          // leader: both CTAs' A and B landed and the copy warps' commits arrived
    uint64_t sf_full[G::kStages];       // leader: both CTAs' scale atoms landed
    uint64_t empty[G::kStages];         // both CTAs, arrived by the leader's commits
    uint64_t acc_full;                  // both CTAs
    uint64_t acc_empty;                 // used in the leader
    uint32_t tmem_base;
};
constexpr size_t kSmemBytes = sizeof(Smem) + 1024;

template <bool kGated>
__global__ void __launch_bounds__(kThreadsPair, 1)
    nvf4_gemm_pair_cp_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                             const __grid_constant__ CUtensorMap tmSFA, const __grid_constant__ CUtensorMap tmSFB,
                             const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmR,
                             const __grid_constant__ GatedEpilogue ge, const float *__restrict__ a_ts,
                             const float *__restrict__ b_ts, int m, int n, int k, int m_tiles2, int n_tiles,
                             int n_group, uint64_t wait_ns, int withhold_loads)
{
    using G = Geo;
    constexpr int kStages = G::kStages;
    extern __shared__ uint8_t smem_raw[];
    Smem &sm = *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const int pair_id = blockIdx.x >> 1, num_pairs = gridDim.x >> 1;
    const int kt_count = k / BK;
    const int sf_rows_per_rb = k / 32;          // 256-byte rows of scale atoms per 128-row block
    const int total_tiles = m_tiles2 * n_tiles;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            // the producer's expect-tx arrival plus one commit per copy warp (scales in TMEM)
            mbar_init(smem_u32(&sm.full[s]), 1 + kCopyWarps);
            mbar_init(smem_u32(&sm.sf_full[s]), 1);
            mbar_init(smem_u32(&sm.empty[s]), 1);
        }
        mbar_init(smem_u32(&sm.acc_full), 1);
        mbar_init(smem_u32(&sm.acc_empty), 2 * kEpiWarps);
        for (int w = 0; w < kEpiWarps; ++w)
            for (int r = 0; r < kResBufs; ++r)
                mbar_init(smem_u32(&sm.res_full[w][r]), 1);
        fence_mbar_init();
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
        prefetch_tmap(&tmSFA);
        prefetch_tmap(&tmSFB);
        prefetch_tmap(&tmC);
        if (kGated)
            prefetch_tmap(&tmR);
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(&sm.tmem_base), TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync();   // barriers of both CTAs initialised, TMEM allocated
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;

    if (warp == 0) {
        // withhold_loads (failure-detection entry point only): no copy is issued,
        // so every wait of the other warps runs out after wait_ns
        if (lane == 0 && !withhold_loads) {
            uint32_t it = 0;
            bool ok = true;
            for (int t = pair_id; t < total_tiles && ok; t += num_pairs) {
                int mt2, nt;
                tile_coords(t, m_tiles2, n_tiles, n_group, mt2, nt);
                const int rb_a = 2 * mt2 + static_cast<int>(rank);
                for (int kt = 0; kt < kt_count; ++kt, ++it) {
                    const int s = it % kStages;
                    if (!mbar_wait_bounded(smem_u32(&sm.empty[s]), ((it / kStages) & 1) ^ 1u, wait_ns)) {
                        record_error(ERR_WAIT_EMPTY);
                        ok = false;
                        break;
                    }
                    if (rank == 0) {
                        mbar_arrive_expect_tx(smem_u32(&sm.sf_full[s]), G::SF_TX);
                        mbar_arrive_expect_tx(smem_u32(&sm.full[s]), G::AB_TX);
                    }
                    // scales first, on their own barrier: the copy warp moves them into TMEM
                    // while A and B are still in flight
                    const uint32_t sbar = mapa_shared(smem_u32(&sm.sf_full[s]), 0);
                    constexpr int sf_stage_rows = G::SFA_BYTES / 256;
                    tma_load_2d_pair(smem_u32(sm.sfa[s]), &tmSFA, 0, rb_a * sf_rows_per_rb + kt * sf_stage_rows, sbar);
                    tma_load_2d_pair(smem_u32(sm.sfb[s]), &tmSFB, 0, 2 * nt * sf_rows_per_rb + kt * sf_stage_rows, sbar);
                    tma_load_2d_pair(smem_u32(sm.sfb[s]) + G::SFB_BYTES / 2, &tmSFB, 0,
                                     (2 * nt + 1) * sf_rows_per_rb + kt * sf_stage_rows, sbar);
                    const uint32_t bar = mapa_shared(smem_u32(&sm.full[s]), 0);
                    tma_load_2d_pair(smem_u32(sm.a[s]), &tmA, kt * G::ROW, mt2 * 256 + static_cast<int>(rank) * 128,
                                     bar);
                    tma_load_2d_pair(smem_u32(sm.b[s]), &tmB, kt * G::ROW, nt * PBN + static_cast<int>(rank) * 128,
                                     bar);
                }
            }
        }
    } else if (warp >= kFirstCopyWarp && warp < kFirstEpi) {
        // Leader only: per stage, wait until both CTAs' scale atoms landed,
        // copy them into both CTAs' TMEM slot for the stage (each CTA's shared
        // memory into its own TMEM) and commit to sf_ready.  The two copy
        // warps split the stage's MMAs between them (6 copies each).  A slot is
        // rewritten only after its stage's scale barrier completed again, i.e.
        // after the producers saw the commit of the MMAs that last read it.
        constexpr int kPerWarp = G::kChunks / kCopyWarps;
        const int j0 = (warp - kFirstCopyWarp) * kPerWarp;
        if (rank == 0) {
            uint32_t it = 0;
            bool ok = true;
            for (int t = pair_id; t < total_tiles && ok; t += num_pairs) {
                for (int kt = 0; kt < kt_count; ++kt, ++it) {
                    const int s = it % kStages;
                    if (!warp_wait(smem_u32(&sm.sf_full[s]), (it / kStages) & 1, wait_ns)) {
                        if (lane == 0)
                            record_error(ERR_WAIT_SCALES);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sfa_t = tmem + SF_COL + s * G::SF_COLS;
                    const uint32_t sfb_t = sfa_t + 4 * G::kChunks;
                    const uint32_t sfa_s = smem_u32(sm.sfa[s]), sfb_s = smem_u32(sm.sfb[s]);
#pragma unroll
                    for (int j = j0; j < j0 + kPerWarp; ++j) {
                        tc_cp_32x128b_warpx4_pair_elect(sfa_t + 4 * j, smem_desc(sfa_s + j * ATOM, 0, 128, 0));
                        tc_cp_32x128b_warpx4_pair_elect(sfb_t + 8 * j, smem_desc(sfb_s + j * ATOM, 0, 128, 0));
                        tc_cp_32x128b_warpx4_pair_elect(sfb_t + 8 * j + 4,
                                                        smem_desc(sfb_s + G::SFB_BYTES / 2 + j * ATOM, 0, 128, 0));
                    }
                    tc_commit_pair_mc_elect(smem_u32(&sm.full[s]), 0x1);
                }
            }
        }
    } else if (warp == 1) {
        // Leader only: per stage, wait for sf_ready (the scales are in TMEM)
        // and full (A and B landed), issue the pair MMAs and commit the stage
        // free in both CTAs.  With the scale copies in their own warp this
        // warp issues 5 tcgen05 instructions per stage instead of 17: its
        // per-stage issue time, which the tensor pipe otherwise waits on,
        // drops well below the MMAs' own time.
        if (rank == 0) {
            constexpr uint32_t idesc = idesc_nvf4(2 * PBM, PBN);
            const int my_tiles = pair_id < total_tiles ? (total_tiles - pair_id + num_pairs - 1) / num_pairs : 0;
            const uint32_t total_steps = static_cast<uint32_t>(my_tiles) * static_cast<uint32_t>(kt_count);
            uint32_t it = 0, local = 0;
            bool ok = true;
            bool known_ready = false;   // the current stage's barrier was seen complete during the previous stage
            for (int t = pair_id; t < total_tiles && ok; t += num_pairs, ++local) {
                if (!warp_wait(smem_u32(&sm.acc_empty), (local & 1) ^ 1u, wait_ns)) {
                    if (lane == 0)
                        record_error(ERR_WAIT_ACC_EMPTY);
                    break;
                }
                tc_fence_after();
                for (int kt = 0; kt < kt_count; ++kt, ++it) {
                    const int s = it % kStages;
                    if (!known_ready && !warp_wait_spin(smem_u32(&sm.full[s]), (it / kStages) & 1, wait_ns)) {
                        if (lane == 0)
                            record_error(ERR_WAIT_FULL);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sfa_t = tmem + SF_COL + s * G::SF_COLS;
                    const uint32_t sfb_t = sfa_t + 4 * G::kChunks;
                    const uint64_t a_desc = smem_desc(smem_u32(sm.a[s]), 0, G::SBO, G::LAYOUT);
                    const uint64_t b_desc = smem_desc(smem_u32(sm.b[s]), 0, G::SBO, G::LAYOUT);
#pragma unroll
                    for (int j = 0; j < kStageMmas - 1; ++j)
                        tc_mma_nvf4_pair_elect(tmem + ACC_COL, a_desc + stage_mma_desc(j), b_desc + stage_mma_desc(j),
                                               stage_mma_idesc(idesc, j), sfa_t + 4 * stage_mma_chunk(j),
                                               sfb_t + 8 * stage_mma_chunk(j), (kt | j) != 0);
                    // While this stage's MMAs run, look (without waiting) whether the next
                    // stage is already complete; if so the next iteration skips its wait,
                    // whose latency otherwise lands between two stages' MMAs.
                    const uint32_t nx = it + 1;
                    known_ready = nx < total_steps &&
                                  __all_sync(0xFFFFFFFFu, mbar_test_wait(smem_u32(&sm.full[nx % kStages]),
                                                                         (nx / kStages) & 1));
                    constexpr int jl = kStageMmas - 1;
                    tc_mma_nvf4_pair_elect(tmem + ACC_COL, a_desc + stage_mma_desc(jl), b_desc + stage_mma_desc(jl),
                                           stage_mma_idesc(idesc, jl), sfa_t + 4 * stage_mma_chunk(jl),
                                           sfb_t + 8 * stage_mma_chunk(jl), 1u);
                    tc_commit_pair_mc_elect(smem_u32(&sm.empty[s]), 0x3);
                }
                if (ok)
                    tc_commit_pair_mc_elect(smem_u32(&sm.acc_full), 0x3);
            }
        }
    } else {
        const int q = warp & 3;
        const int half = (warp - kFirstEpi) >> 2;
        const float alpha = __fmul_rn(*a_ts, *b_ts);
        const uint32_t leader_acc_empty = mapa_shared(smem_u32(&sm.acc_empty), 0);
        uint32_t local = 0, rphase = 0;
        for (int t = pair_id; t < total_tiles; t += num_pairs, ++local) {
            int mt2, nt;
            tile_coords(t, m_tiles2, n_tiles, n_group, mt2, nt);
            if (!warp_wait(smem_u32(&sm.acc_full), local & 1, wait_ns)) {
                if (lane == 0)
                    record_error(ERR_WAIT_ACC);
                break;
            }
            tc_fence_after();
            uint32_t pk[64];
            const uint32_t base = tmem + (static_cast<uint32_t>(q * 32) << 16) + ACC_COL + half * 128;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t v[32];
                tmem_ld_32x32b_x32(base + 32 * c, v);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float lo = __fmul_rn(alpha, __uint_as_float(v[2 * i]));
                    const float hi = __fmul_rn(alpha, __uint_as_float(v[2 * i + 1]));
                    const __nv_bfloat162 b2 = __floats2bfloat162_rn(lo, hi);
                    memcpy(&pk[16 * c + i], &b2, 4);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)   // this CTA's rows are drained (relaxed: earlier tiles' stores need not land first)
                mbar_arrive_cluster_relaxed(leader_acc_empty);
            const int row0 = mt2 * 256 + static_cast<int>(rank) * PBM + q * 32;
            if (kGated) {
                if (!store_rows_gated_ring<kResBufs>(&tmC, &tmR, smem_u32(sm.cst[warp - kFirstEpi][0]),
                                                     smem_u32(&sm.res_full[warp - kFirstEpi][0]), rphase, pk,
                                                     nt * PBN + half * 128, row0, lane,
                                                     gate_row(ge, row0 + lane))) {
                    if (lane == 0)
                        record_error(ERR_WAIT_ACC);
                    break;
                }
            } else {
                store_rows(&tmC, smem_u32(sm.cst[warp - kFirstEpi][0]), pk, nt * PBN + half * 128, row0, lane);
            }
        }
        if (lane == 0)
            bulk_wait_group0();
    }

    tc_fence_before();
    cluster_sync();   // no CTA leaves while its peer may still touch its barriers or TMEM
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, TMEM_COLS);
    }
}

}  // namespace paircp


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

// 2-D bf16 tensor map over the output C [m, n] with row stride ldc elements,
// box 16 columns x 32 rows (one epilogue warp's store), no swizzle.
bool make_output_map(CUtensorMap *tm, void *base, int64_t m, int64_t n, int64_t ldc)
{
    auto fn = encode_fn();
    if (!fn)
        return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(n), static_cast<cuuint64_t>(m)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ldc * 2)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(CST_COLS), 32};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 2-D uint8 tensor map viewing a scale buffer of `bytes` bytes as rows of 256
// bytes, box 256 x 8 (one 2 KB chunk = 4 scale atoms), no swizzle.
bool make_scale_map(CUtensorMap *tm, const void *base, int64_t bytes)
{
    auto fn = encode_fn();
    if (!fn)
        return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(paircp::SF_ROW), static_cast<cuuint64_t>(bytes / paircp::SF_ROW)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(paircp::SF_ROW)};
    cuuint32_t box[2] = {paircp::SF_ROW, 8};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace

namespace {

template <bool kGated>
h3fp4_status launch_tiles(const CUtensorMap &tmA, const CUtensorMap &tmB, const CUtensorMap &tmC, const CUtensorMap &tmR,
                          const GatedEpilogue &ge, const uint8_t *a_sf, const uint8_t *b_sf, const float *a_ts,
                          const float *b_ts, int64_t m, int64_t n, int64_t k, int n_group_cfg, cudaStream_t st)
{
    static bool attr_set[64] = {false};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return H3FP4_ERR_CUDA;
    if (dev >= 0 && dev < 64 && !attr_set[dev]) {
        if (cudaFuncSetAttribute(nvf4_gemm_kernel<kGated>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kSmemBytes)) != cudaSuccess)
            return H3FP4_ERR_CUDA;
        attr_set[dev] = true;
    }
    const int m_tiles = static_cast<int>((m + BM - 1) / BM);
    const int n_tiles = static_cast<int>((n + BN - 1) / BN);
    const int64_t total = static_cast<int64_t>(m_tiles) * n_tiles;
    if (total > 0x7FFFFFFF)
        return H3FP4_ERR_SHAPE;
    int n_group = n_group_cfg > 0 ? n_group_cfg : kDefaultNGroup;
    if (n_group > n_tiles)
        n_group = n_tiles;
    const int grid = static_cast<int>(total < sm_count() ? total : sm_count());
    nvf4_gemm_kernel<kGated><<<grid, kThreads, kSmemBytes, st>>>(tmA, tmB, tmC, tmR, ge, a_sf, b_sf, a_ts, b_ts,
                                                                 static_cast<int>(m), static_cast<int>(n),
                                                                 static_cast<int>(k), m_tiles, n_tiles, n_group);
    return cudaGetLastError() == cudaSuccess ? H3FP4_OK : H3FP4_ERR_CUDA;
}

}  // namespace

// Tensor map of the residual and the kernel-parameter copy of the gate
// arguments (both unused without a gated epilogue).
bool make_gated(const GatedArgs *gated, const CUtensorMap &tmC, int64_t m, int64_t n, CUtensorMap *tmR,
                GatedEpilogue *ge)
{
    *ge = GatedEpilogue{};
    if (gated == nullptr) {
        *tmR = tmC;
        return true;
    }
    if (!make_output_map(tmR, const_cast<void *>(gated->residual), m, n, gated->ldr))
        return false;
    ge->gate = gated->gate;
    ge->ld_gate = gated->ld_gate;
    for (int i = 0; i <= H3FP4_MAX_SEGMENTS; ++i)
        ge->off[i] = gated->seg.off[i];
    ge->nseg = gated->seg.nseg;
    return true;
}

template <bool kGated>
cudaError_t set_pair_cp_smem()
{
    static bool attr_set[64] = {false};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev >= 0 && dev < 64 && !attr_set[dev]) {
        e = cudaFuncSetAttribute(paircp::nvf4_gemm_pair_cp_kernel<kGated>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(paircp::kSmemBytes));
        if (e != cudaSuccess)
            return e;
        attr_set[dev] = true;
    }
    return cudaSuccess;
}

// Default N-group of the CTA-pair kernel: the fewest near-equal groups of
// N-tiles whose B tiles (256 rows x k/2 bytes each) stay within ~27.5 MB, the
// set that must stay L2-resident while a group sweeps all M tiles.  Measured
// at 37,810 rows: k = 7,168 -> 28 of 84 or 56 tiles, k = 14,336 -> 14 of 28
// (8 % faster than 28) and 11 of 21, k = 5,376 -> 28 of 84.
int pair_default_n_group(int n_tiles, int64_t k)
{
    const int64_t target = 27500000 / (128 * k) > 1 ? 27500000 / (128 * k) : 1;
    const int64_t groups = (n_tiles + target - 1) / target;
    return static_cast<int>((n_tiles + groups - 1) / groups);
}

h3fp4_status launch_pair_cp(const uint8_t *a_q, const uint8_t *a_sf, const float *a_ts, const uint8_t *b_q,
                            const uint8_t *b_sf, const float *b_ts, uint16_t *c, int64_t ldc, int64_t m,
                            int64_t m_pad, int64_t n, int64_t k, int n_group_cfg, const GatedArgs *gated,
                            cudaStream_t st, uint64_t wait_ns = kWaitLimitNs, int withhold_loads = 0)
{
    const int64_t sfa_rows = (m_pad + 127) / 128 * 128, sfb_rows = (n + 127) / 128 * 128;
    CUtensorMap tmA, tmB, tmSFA, tmSFB, tmC, tmR;
    GatedEpilogue ge;
    if (!make_operand_map(&tmA, a_q, m_pad, k / 2, paircp::PBM) || !make_operand_map(&tmB, b_q, n, k / 2, 128) ||
        !make_scale_map(&tmSFA, a_sf, sfa_rows * (k / 16)) || !make_scale_map(&tmSFB, b_sf, sfb_rows * (k / 16)) ||
        !make_output_map(&tmC, c, m, n, ldc) || !make_gated(gated, tmC, m, n, &tmR, &ge))
        return H3FP4_ERR_CUDA;
    if ((gated ? set_pair_cp_smem<true>() : set_pair_cp_smem<false>()) != cudaSuccess)
        return H3FP4_ERR_CUDA;
    const int m_tiles2 = static_cast<int>((m + 255) / 256);
    const int n_tiles = static_cast<int>((n + paircp::PBN - 1) / paircp::PBN);
    const int64_t total = static_cast<int64_t>(m_tiles2) * n_tiles;
    if (total > 0x7FFFFFFF)
        return H3FP4_ERR_SHAPE;
    int n_group = n_group_cfg > 0 ? n_group_cfg : pair_default_n_group(n_tiles, k);
    if (n_group > n_tiles)
        n_group = n_tiles;
    const int max_pairs = sm_count() / 2;
    const int pairs = static_cast<int>(total < max_pairs ? total : max_pairs);
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(2 * pairs, 1, 1);
    lc.blockDim = dim3(paircp::kThreadsPair, 1, 1);
    lc.dynamicSmemBytes = paircp::kSmemBytes;
    lc.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    const cudaError_t e =
        gated ? cudaLaunchKernelEx(&lc, paircp::nvf4_gemm_pair_cp_kernel<true>, tmA, tmB, tmSFA, tmSFB, tmC, tmR,
                                   ge, a_ts, b_ts, static_cast<int>(m), static_cast<int>(n), static_cast<int>(k),
                                   m_tiles2, n_tiles, n_group, wait_ns, withhold_loads)
              : cudaLaunchKernelEx(&lc, paircp::nvf4_gemm_pair_cp_kernel<false>, tmA, tmB, tmSFA, tmSFB, tmC, tmR, ge,
                                   a_ts, b_ts, static_cast<int>(m), static_cast<int>(n), static_cast<int>(k), m_tiles2,
                                   n_tiles, n_group, wait_ns, withhold_loads);
    return e == cudaSuccess ? H3FP4_OK : H3FP4_ERR_CUDA;
}

h3fp4_status launch_gemm(const uint8_t *a_q, const uint8_t *a_sf, const float *a_ts, const uint8_t *b_q,
                         const uint8_t *b_sf, const float *b_ts, uint16_t *c, int64_t ldc, int64_t m, int64_t m_pad,
                         int64_t n, int64_t k, const h3fp4_gemm_config &cfg, const GatedArgs *gated, cudaStream_t st)
{
    if (m == 0 || n == 0)
        return H3FP4_OK;
    if (cfg.cta_pair == 0 || cfg.cta_pair == 4)   // the default: measured fastest in the DiT step
        return launch_pair_cp(a_q, a_sf, a_ts, b_q, b_sf, b_ts, c, ldc, m, m_pad, n, k, cfg.n_group, gated, st);
    if (cfg.cta_pair != 1)
        return H3FP4_ERR_UNSUPPORTED;
    CUtensorMap tmA, tmB, tmC, tmR;
    GatedEpilogue ge;
    if (!make_operand_map(&tmA, a_q, m_pad, k / 2, BM) || !make_operand_map(&tmB, b_q, n, k / 2, BN) ||
        !make_output_map(&tmC, c, m, n, ldc) || !make_gated(gated, tmC, m, n, &tmR, &ge))
        return H3FP4_ERR_CUDA;
    return gated ? launch_tiles<true>(tmA, tmB, tmC, tmR, ge, a_sf, b_sf, a_ts, b_ts, m, n, k, cfg.n_group, st)
                 : launch_tiles<false>(tmA, tmB, tmC, tmR, ge, a_sf, b_sf, a_ts, b_ts, m, n, k, cfg.n_group, st);
}

h3fp4_status launch_gemm_wait_timeout(const uint8_t *a_q, const uint8_t *a_sf, const float *a_ts,
                                      const uint8_t *b_q, const uint8_t *b_sf, const float *b_ts, uint16_t *c,
                                      int64_t ldc, int64_t m, int64_t m_pad, int64_t n, int64_t k, uint64_t wait_ns,
                                      cudaStream_t st)
{
    if (m == 0 || n == 0)
        return H3FP4_OK;
    return launch_pair_cp(a_q, a_sf, a_ts, b_q, b_sf, b_ts, c, ldc, m, m_pad, n, k, 0, nullptr, st, wait_ns, 1);
}

h3fp4_status read_device_error(uint32_t *code)
{
    uint32_t v = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v)) != cudaSuccess)
        return H3FP4_ERR_CUDA;
    const uint32_t zero = 0;
    if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero)) != cudaSuccess)
        return H3FP4_ERR_CUDA;
    uint32_t p = 0;
    if (read_producer_error(&p) != cudaSuccess)
        return H3FP4_ERR_CUDA;
    *code = v | p;
    return H3FP4_OK;
}

}  // namespace h3fp4
