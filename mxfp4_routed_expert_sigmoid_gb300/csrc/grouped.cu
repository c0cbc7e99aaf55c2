// tcgen05 GEMMs: the grouped expert GEMMs of the routed layer and the dense
// bf16 GEMM used for the latent projections and the router at large T.
//
// One persistent, warp-specialised kernel template computes
//     D[m, n] = sum_c A[m, c] * B[n, c]       (A: weights, B: token rows)
// with M = 128 weight rows per tile (TMEM lanes), N = up to BN token rows
// per tile (TMEM columns, fp32), K in stages of 64 (128 bytes of f16/bf16
// per row: the 128-byte swizzled K-major shared-memory layout of tcgen05).
//
// Roles (warps):
//   0      producer: TMA loads of B (tokens) and of A (dense mode) or of the
//          raw MXFP4 bytes of A (expert modes) into a ring of stages;
//   1      MMA issuer: one thread issues tcgen05.mma kind::f16 per 16-wide K
//          slice and commits each stage back to the producer;
//   2      TMEM allocation / release;
//   4..7   epilogue: tcgen05.ld of the fp32 accumulator (lane = weight row),
//          scaling, activation and stores (coalesced along the weight rows);
//   8..15  dequantisation (expert modes): E2M1 codes -> f16 (hardware cvt),
//          times the block scale 2^(e - e_ref) in f16, written into the
//          swizzled A stage.  e_ref is the largest exponent of the weight row,
//          applied in fp32 by the epilogue as 2^(e_ref - 127) (exact).
// Accumulators are double buffered in TMEM so the epilogue of one tile runs
// under the main loop of the next.
//
// Expert modes (llama.cpp PR #26185 "model: add Kimi-K3 text model": latent
// MoE; w1/w3 logical [f, d], w2 [d, f], MXFP4 blocks of 32 along the input):
//   UP   : A = W1 and W3 rows of expert e, B = the expert's gathered token
//          rows (f16, one power-of-two exponent per row); epilogue h =
//          silu(g) * u, stored fp32 with a per-row |h| maximum;
//   DOWN : A = W2 rows, B = the f16 h rows; epilogue y in fp32.
// Work units (expert, first row, row count <= BN) are built on the device
// from the permutation, so no token count ever returns to the host.
//
// Every mbarrier wait is bounded (2 s); on expiry the kernel records
// K3MOE_ERR_TIMEOUT in the workspace status word, all roles drain, TMEM is
// released and the kernel returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "common.cuh"

namespace k3 {
namespace {

enum Mode { DENSE = 0, UP = 1, DOWN = 2 };

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int kTileA = BM * BK * 2;   // 16 KB of f16/bf16
constexpr int kTileRaw = BM * BK / 2; // 4 KB of packed E2M1

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait: false if the CTA is aborting or the limit expired.
__device__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, WsHeader* hdr,
                          int where) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (global_ns() - t0 > kWaitLimitNs) {
            *abort_flag = 1;
            if (hdr) set_error(hdr, K3MOE_ERR_TIMEOUT, where);
            return false;
        }
    }
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* tm, uint64_t* bar, int x,
                                            int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(smem_u32(bar)), "r"(x), "r"(y)
        : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* tm) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tm)) : "memory");
}

__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);  // start address
    d |= static_cast<uint64_t>(1) << 16;                    // leading byte offset (unused here)
    d |= static_cast<uint64_t>(1024 >> 4) << 32;            // stride byte offset
    d |= static_cast<uint64_t>(1) << 46;                    // descriptor version
    d |= static_cast<uint64_t>(2) << 61;                    // 128-byte swizzle
    return d;
}

// Instruction descriptor, kind::f16: fp32 accumulator, A/B f16 (fmt 0) or
// bf16 (fmt 1), both K-major, shape M x N.
__device__ __forceinline__ uint32_t idesc_f16(int fmt, int M, int N) {
    return (1u << 4) | (static_cast<uint32_t>(fmt) << 7) | (static_cast<uint32_t>(fmt) << 10) |
           (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// ---------------------------------------------------------------------------
// kernel parameters
// ---------------------------------------------------------------------------
struct TcParams {
    int K;                 // reduction length (multiple of 64)
    int rows_per_expert;   // expert modes: rows of one expert matrix (f or d)
    int m_tiles;           // 128-row tiles per expert matrix (or over N_out in dense mode)
    int T;                 // dense: token rows
    int n_tiles;           // dense: token tiles
    const uint8_t* s1;     // expert: E8M0 scales of A (w1 or w2), [E * rows, K / 32]
    const uint8_t* s3;     // UP: scales of w3
    const int4* units;     // expert: units[0].x = count; units[1 + u] = (e, row0, nrows, 0)
    const int32_t* bexp;   // expert: per B row power-of-two exponent
    void* out;             // dense: [T, N_out] bf16 or fp32
    int out_fp32;
    int n_out;             // dense: N_out (row length of out); expert: width of hb / y rows
    float* hf;             // UP: h in fp32 [P, f]
    uint32_t* h_amax;      // UP: max |h| per row (fp32 bits)
    float* y;              // DOWN: [P, d]
    WsHeader* hdr;
};

template <int MODE>
struct Cfg;
template <>
struct Cfg<DENSE> {
    static constexpr int NA = 1, BN = 256, STAGES = 4, THREADS = 256, TMEM_COLS = 512;
};
template <>
struct Cfg<UP> {
    static constexpr int NA = 2, BN = 128, STAGES = 3, THREADS = 512, TMEM_COLS = 512;
};
template <>
struct Cfg<DOWN> {
    static constexpr int NA = 1, BN = 128, STAGES = 4, THREADS = 512, TMEM_COLS = 256;
};

template <int MODE>
constexpr size_t smem_bytes() {
    using C = Cfg<MODE>;
    size_t b = 1024;  // alignment slack
    b += static_cast<size_t>(C::STAGES) * C::NA * kTileA;
    b += static_cast<size_t>(C::STAGES) * C::BN * BK * 2;
    if (MODE != DENSE) b += static_cast<size_t>(C::STAGES) * C::NA * kTileRaw;
    b += 256;  // barriers, flags
    return b;
}

__device__ __forceinline__ float silu_f32(float g) { return g / (1.0f + expf(-g)); }

// largest E8M0 exponent of a weight row of nb bytes (16-byte loads when the
// row length allows it; rows are then 16-byte aligned because the scale
// array is)
__device__ __forceinline__ int row_emax(const uint8_t* srow, int nb) {
    int m = 0;
    if ((nb & 15) == 0) {
        for (int i = 0; i < nb; i += 16) {
            const uint4 v = *reinterpret_cast<const uint4*>(srow + i);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int b = 0; b < 4; ++b) m = max(m, static_cast<int>((w[j] >> (8 * b)) & 0xFF));
        }
    } else {
        for (int i = 0; i < nb; ++i) m = max(m, static_cast<int>(srow[i]));
    }
    return m;
}

// tile -> (expert, first B row, B rows, m tile); returns false past the end
template <int MODE>
__device__ __forceinline__ bool tile_info(const TcParams& p, int tile, int n_tiles, int& e,
                                          int& row0, int& nrows, int& mt) {
    if (tile >= n_tiles) return false;
    mt = tile % p.m_tiles;
    const int u = tile / p.m_tiles;
    if (MODE == DENSE) {
        e = 0;
        row0 = u * Cfg<DENSE>::BN;
        nrows = min(Cfg<DENSE>::BN, p.T - row0);
    } else {
        const int4 un = p.units[1 + u];
        e = un.x;
        row0 = un.y;
        nrows = un.z;
    }
    return true;
}

template <int MODE>
__global__ void __launch_bounds__(Cfg<MODE>::THREADS, 1)
tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA3,
               const __grid_constant__ CUtensorMap tmB, TcParams p) {
    using C = Cfg<MODE>;
    constexpr int NA = C::NA, BN = C::BN, STAGES = C::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;                                          // [STAGES][NA][16 KB]
    uint8_t* sB = sA + STAGES * NA * kTileA;                     // [STAGES][BN * 128]
    uint8_t* sRaw = sB + STAGES * BN * BK * 2;                   // [STAGES][NA][4 KB]
    uint8_t* tail = sRaw + (MODE != DENSE ? STAGES * NA * kTileRaw : 0);
    uint64_t* full_b = reinterpret_cast<uint64_t*>(tail);        // TMA B (+A in dense mode)
    uint64_t* full_raw = full_b + STAGES;                        // TMA raw A
    uint64_t* full_a = full_raw + STAGES;                        // dequantised A ready
    uint64_t* empty = full_a + STAGES;                           // MMA done with stage
    uint64_t* acc_full = empty + STAGES;                         // [2]
    uint64_t* acc_empty = acc_full + 2;                          // [2]
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(acc_empty + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_tiles = (MODE == DENSE) ? p.n_tiles * p.m_tiles : p.units[0].x * p.m_tiles;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full_b[s], 1);
            mbar_init(&full_raw[s], 1);
            mbar_init(&full_a[s], 8);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&acc_full[a], 1);
            mbar_init(&acc_empty[a], 4);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        fence_proxy_async();
    }
    if (warp == 2) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_holder)),
                     "r"(C::TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
        if (MODE == UP) prefetch_tmap(&tmA3);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    const int k_stages = p.K / BK;

    if (warp == 0) {
        // ------------------------------ producer ------------------------------
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            for (int tile = blockIdx.x;; tile += gridDim.x) {
                int e, row0, nrows, mt;
                if (!tile_info<MODE>(p, tile, n_tiles, e, row0, nrows, mt)) break;
                const int arow = (MODE == DENSE) ? mt * BM : e * p.rows_per_expert + mt * BM;
                bool ok = true;
                for (int ks = 0; ks < k_stages; ++ks) {
                    if (!mbar_wait(&empty[s], ph ^ 1, abort_flag, p.hdr, 10)) { ok = false; break; }
                    if (MODE == DENSE) {
                        mbar_expect_tx(&full_b[s], kTileA + BN * BK * 2);
                        tma_load_2d(sA + s * kTileA, &tmA, &full_b[s], ks * BK, arow);
                        tma_load_2d(sB + s * BN * BK * 2, &tmB, &full_b[s], ks * BK, row0);
                    } else {
                        mbar_expect_tx(&full_raw[s], NA * kTileRaw);
                        tma_load_2d(sRaw + (s * NA) * kTileRaw, &tmA, &full_raw[s], ks * BK / 2, arow);
                        if (MODE == UP)
                            tma_load_2d(sRaw + (s * NA + 1) * kTileRaw, &tmA3, &full_raw[s], ks * BK / 2,
                                        arow);
                        mbar_expect_tx(&full_b[s], BN * BK * 2);
                        tma_load_2d(sB + s * BN * BK * 2, &tmB, &full_b[s], ks * BK, row0);
                    }
                    if (++s == STAGES) { s = 0; ph ^= 1; }
                }
                if (!ok) break;
            }
        }
    } else if (warp == 1) {
        // ------------------------------ MMA issuer ----------------------------
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            int it = 0;
            const int fmt = (MODE == DENSE) ? 1 : 0;
            for (int tile = blockIdx.x;; tile += gridDim.x, ++it) {
                int e, row0, nrows, mt;
                if (!tile_info<MODE>(p, tile, n_tiles, e, row0, nrows, mt)) break;
                const int acc = it & 1;
                const uint32_t acc_ph = (it >> 1) & 1;
                const int n_mma = (MODE == DENSE) ? BN : ((nrows + 15) / 16) * 16;
                const uint32_t idesc = idesc_f16(fmt, BM, n_mma);
                if (!mbar_wait(&acc_empty[acc], acc_ph ^ 1, abort_flag, p.hdr, 20)) break;
                tc_fence_after();
                const uint32_t d0 = tmem_base + static_cast<uint32_t>(acc * NA * BN);
                bool ok = true;
                for (int ks = 0; ks < k_stages; ++ks) {
                    if (!mbar_wait(&full_b[s], ph, abort_flag, p.hdr, 21)) { ok = false; break; }
                    if (MODE != DENSE && !mbar_wait(&full_a[s], ph, abort_flag, p.hdr, 22)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t b_addr = smem_u32(sB + s * BN * BK * 2);
#pragma unroll
                    for (int a = 0; a < NA; ++a) {
                        const uint32_t a_addr = smem_u32(sA + (s * NA + a) * kTileA);
#pragma unroll
                        for (int kk = 0; kk < BK / 16; ++kk)
                            mma_f16(d0 + a * BN, sw128_desc(a_addr + kk * 32), sw128_desc(b_addr + kk * 32),
                                    idesc, (ks > 0 || kk > 0) ? 1u : 0u);
                    }
                    mma_commit(&empty[s]);
                    if (++s == STAGES) { s = 0; ph ^= 1; }
                }
                if (!ok) break;
                mma_commit(&acc_full[acc]);
            }
        }
    } else if (warp >= 4 && warp < 8) {
        // ------------------------------ epilogue ------------------------------
        const int wr = warp & 3;
        const int m = wr * 32 + lane;  // accumulator lane = weight row in the tile
        int it = 0;
        for (int tile = blockIdx.x;; tile += gridDim.x, ++it) {
            int e, row0, nrows, mt;
            if (!tile_info<MODE>(p, tile, n_tiles, e, row0, nrows, mt)) break;
            const int acc = it & 1;
            const uint32_t acc_ph = (it >> 1) & 1;
            if (!__all_sync(0xffffffffu, mbar_wait(&acc_full[acc], acc_ph, abort_flag, p.hdr, 30)))
                break;
            tc_fence_after();
            const uint32_t tbase = tmem_base + (static_cast<uint32_t>(wr * 32) << 16) +
                                   static_cast<uint32_t>(acc * NA * BN);
            const int n_used = (MODE == DENSE) ? BN : ((nrows + 15) / 16) * 16;
            if (MODE == DENSE) {
                const int col = mt * BM + m;  // output feature
                for (int n0 = 0; n0 < n_used; n0 += 16) {
                    float v[16];
                    tmem_ld16(tbase + n0, v);
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int t = row0 + n0 + i;
                        if (n0 + i < nrows) {
                            if (p.out_fp32)
                                static_cast<float*>(p.out)[static_cast<size_t>(t) * p.n_out + col] = v[i];
                            else
                                static_cast<uint16_t*>(p.out)[static_cast<size_t>(t) * p.n_out + col] =
                                    f32_to_bf16(v[i]);
                        }
                    }
                }
            } else {
                const int r = mt * BM + m;  // row of the expert matrix
                const bool valid = r < p.rows_per_expert;
                const int nb = p.K / 32;
                const size_t srow = (static_cast<size_t>(e) * p.rows_per_expert + (valid ? r : 0)) * nb;
                const int eref1 = row_emax(p.s1 + srow, nb);
                const int eref3 = (MODE == UP) ? row_emax(p.s3 + srow, nb) : 0;
                for (int n0 = 0; n0 < n_used; n0 += 16) {
                    float v1[16];
                    tmem_ld16(tbase + n0, v1);
                    if (MODE == UP) {
                        float v3[16];
                        tmem_ld16(tbase + BN + n0, v3);
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            if (n0 + i >= nrows) break;
                            const int pr = row0 + n0 + i;
                            const int xe = p.bexp[pr];
                            const float g = v1[i] * exp2i(eref1 - 127 + xe);
                            const float u = v3[i] * exp2i(eref3 - 127 + xe);
                            const float h = silu_f32(g) * u;
                            if (valid) p.hf[static_cast<size_t>(pr) * p.n_out + r] = h;
                            const float a = warp_max(valid ? fabsf(h) : 0.0f);
                            if (lane == 0) atomicMax(p.h_amax + pr, __float_as_uint(a));
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            if (n0 + i >= nrows) break;
                            const int pr = row0 + n0 + i;
                            const float y = v1[i] * exp2i(eref1 - 127 + p.bexp[pr]);
                            if (valid) p.y[static_cast<size_t>(pr) * p.n_out + r] = y;
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[acc]);
        }
    } else if (MODE != DENSE && warp >= 8) {
        // ------------------------------ dequantisation ------------------------
        const int dt = threadIdx.x - 256;  // 0..255
        const int row = dt >> 1, half = dt & 1;
        const int nb = p.K / 32;
        int s = 0;
        uint32_t ph = 0;
        for (int tile = blockIdx.x;; tile += gridDim.x) {
            int e, row0, nrows, mt;
            if (!tile_info<MODE>(p, tile, n_tiles, e, row0, nrows, mt)) break;
            int r = mt * BM + row;
            if (r >= p.rows_per_expert) r = p.rows_per_expert - 1;  // padding rows: any finite data
            const size_t srow = (static_cast<size_t>(e) * p.rows_per_expert + r) * nb;
            const uint8_t* sc1 = p.s1 + srow;
            const uint8_t* sc3 = (MODE == UP) ? p.s3 + srow : nullptr;
            const int eref1 = row_emax(sc1, nb);
            const int eref3 = (MODE == UP) ? row_emax(sc3, nb) : 0;
            bool ok = true;
            for (int ks = 0; ks < k_stages; ++ks) {
                const int blk = 2 * ks + half;
                const int e1 = sc1[blk];
                const int e3 = (MODE == UP) ? sc3[blk] : 0;
                if (!__all_sync(0xffffffffu, mbar_wait(&full_raw[s], ph, abort_flag, p.hdr, 40))) {
                    ok = false;
                    break;
                }
#pragma unroll
                for (int a = 0; a < NA; ++a) {
                    const uint4 raw =
                        *reinterpret_cast<const uint4*>(sRaw + (s * NA + a) * kTileRaw + row * 32 + half * 16);
                    const uint16_t sh = f16_pow2((a == 0 ? e1 - eref1 : e3 - eref3));
                    const uint32_t sc2 = static_cast<uint32_t>(sh) | (static_cast<uint32_t>(sh) << 16);
                    uint32_t w[16];
                    e2m1x8_to_f16x8(raw.x, w[0], w[1], w[2], w[3]);
                    e2m1x8_to_f16x8(raw.y, w[4], w[5], w[6], w[7]);
                    e2m1x8_to_f16x8(raw.z, w[8], w[9], w[10], w[11]);
                    e2m1x8_to_f16x8(raw.w, w[12], w[13], w[14], w[15]);
#pragma unroll
                    for (int i = 0; i < 16; ++i) w[i] = hmul2(w[i], sc2);
                    uint8_t* dst = sA + (s * NA + a) * kTileA + row * 128;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int chunk = (half * 4 + c) ^ (row & 7);
                        *reinterpret_cast<uint4*>(dst + chunk * 16) =
                            make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
                    }
                }
                fence_proxy_async();
                __syncwarp();
                if (lane == 0) mbar_arrive(&full_a[s]);
                if (++s == STAGES) { s = 0; ph ^= 1; }
            }
            if (!ok) break;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                     "r"(C::TMEM_COLS));
    }
}

// ---------------------------------------------------------------------------
// helper kernels of the grouped path
// ---------------------------------------------------------------------------
// xp[r] = f16(x[token(r)] * 2^-ex), ex = floor(log2(max |x[token(r)]|)); one
// warp per permuted row; also clears h_amax[r].
__global__ void __launch_bounds__(256)
gather_rows_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ perm, int P, int k,
                   int d, uint16_t* __restrict__ xp, int32_t* __restrict__ xexp,
                   uint32_t* __restrict__ h_amax) {
    const int r = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (r >= P) return;
    const int t = perm[r] / k;
    const uint16_t* src = x + static_cast<size_t>(t) * d;
    float amax = 0.0f;
    for (int c = lane * 8; c < d; c += 256) {
        const uint4 v = *reinterpret_cast<const uint4*>(src + c);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
            amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(w[j] << 16)),
                                     fabsf(__uint_as_float(w[j] & 0xFFFF0000u))));
    }
    amax = warp_max(amax);
    const int ex = ilog2f(amax);
    const float sc = exp2i(-ex);
    uint16_t* dst = xp + static_cast<size_t>(r) * d;
    for (int c = lane * 8; c < d; c += 256) {
        const uint4 v = *reinterpret_cast<const uint4*>(src + c);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint4 o;
        uint32_t* oo = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
        for (int j = 0; j < 4; ++j)
            oo[j] = f32x2_to_f16x2(__uint_as_float(w[j] << 16) * sc,
                                   __uint_as_float(w[j] & 0xFFFF0000u) * sc);
        *reinterpret_cast<uint4*>(dst + c) = o;
    }
    if (lane == 0) {
        xexp[r] = ex;
        h_amax[r] = 0u;
    }
}

// hp[r] = f16(hf[r] * 2^-ex), ex = floor(log2(h_amax[r])); one warp per row
__global__ void __launch_bounds__(256)
convert_h_kernel(const float* __restrict__ hf, const uint32_t* __restrict__ h_amax, int P, int f,
                 uint16_t* __restrict__ hp, int32_t* __restrict__ hexp) {
    const int r = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (r >= P) return;
    const int ex = ilog2f(__uint_as_float(h_amax[r]));
    const float sc = exp2i(-ex);
    const float* src = hf + static_cast<size_t>(r) * f;
    uint16_t* dst = hp + static_cast<size_t>(r) * f;
    for (int c = lane * 8; c < f; c += 256) {
        const float4 a = *reinterpret_cast<const float4*>(src + c);
        const float4 b = *reinterpret_cast<const float4*>(src + c + 4);
        uint4 o;
        o.x = f32x2_to_f16x2(a.x * sc, a.y * sc);
        o.y = f32x2_to_f16x2(a.z * sc, a.w * sc);
        o.z = f32x2_to_f16x2(b.x * sc, b.y * sc);
        o.w = f32x2_to_f16x2(b.z * sc, b.w * sc);
        *reinterpret_cast<uint4*>(dst + c) = o;
    }
    if (lane == 0) hexp[r] = ex;
}

// units of at most bn rows per expert: units[0].x = count, units[1 + u] = (e, row0, nrows, 0)
__global__ void __launch_bounds__(256)
build_units_kernel(const int32_t* __restrict__ counts, const int32_t* __restrict__ offsets, int E,
                   int bn, int4* units, int cap) {
    __shared__ int base[1024 + 1];
    for (int e = threadIdx.x; e < E; e += blockDim.x) base[e] = (counts[e] + bn - 1) / bn;
    __syncthreads();
    if (threadIdx.x == 0) {
        int run = 0;
        for (int e = 0; e < E; ++e) {
            const int c = base[e];
            base[e] = run;
            run += c;
        }
        base[E] = run;
        units[0] = make_int4(min(run, cap), 0, 0, 0);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        const int cnt = counts[e];
        for (int c = 0; c * bn < cnt; ++c) {
            const int u = base[e] + c;
            if (u < cap) units[1 + u] = make_int4(e, offsets[e] + c * bn, min(bn, cnt - c * bn), 0);
        }
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// 2-D tensor map over a row-major [outer, inner] array
bool make_tmap(CUtensorMap* tm, const void* base, CUtensorMapDataType dt, int elem_bytes,
               uint64_t inner, uint64_t outer, uint32_t box_inner, uint32_t box_outer,
               CUtensorMapSwizzle sw) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner * static_cast<uint64_t>(elem_bytes)};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(tm, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int MODE>
cudaError_t launch_tc(const CUtensorMap& a, const CUtensorMap& a3, const CUtensorMap& b,
                      const TcParams& p, int grid, cudaStream_t s, const char* name) {
    constexpr size_t smem = smem_bytes<MODE>();
    static_assert(smem <= 232448, "shared memory budget");
    // the attribute is per device; set it once per device (not inside graph captures)
    static std::atomic<uint64_t> done{0};
    int dev = 0;
    cudaGetDevice(&dev);
    const uint64_t bit = 1ull << (dev & 63);
    if (!(done.load() & bit)) {
        cudaError_t e = cudaFuncSetAttribute(tc_gemm_kernel<MODE>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        done.fetch_or(bit);
    }
    tc_gemm_kernel<MODE><<<grid, Cfg<MODE>::THREADS, smem, s>>>(a, a3, b, p);
    trace_mark(name, s);
    return cudaGetLastError();
}

constexpr int kUnitRows = 128;  // == Cfg<UP>::BN == Cfg<DOWN>::BN

}  // namespace

size_t grouped_tile_cap(int T, int E, int k) {
    return static_cast<size_t>(E) + (static_cast<size_t>(T) * k + 15) / 16 + 2;
}

cudaError_t launch_gemm_bf16(const uint16_t* x, const uint16_t* w, int T, int N, int K, void* out,
                             int out_fp32, WsHeader* hdr, int num_sms, cudaStream_t s) {
    if (N % BM || K % BK || T < 1) return cudaErrorInvalidValue;
    CUtensorMap ta, tb;
    if (!make_tmap(&ta, w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, K, N, BK, BM,
                   CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorNotSupported;
    if (!make_tmap(&tb, x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, K, T, BK, Cfg<DENSE>::BN,
                   CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorNotSupported;
    TcParams p{};
    p.K = K;
    p.m_tiles = N / BM;
    p.T = T;
    p.n_tiles = (T + Cfg<DENSE>::BN - 1) / Cfg<DENSE>::BN;
    p.out = out;
    p.out_fp32 = out_fp32;
    p.n_out = N;
    p.hdr = hdr;
    const int tiles = p.n_tiles * p.m_tiles;
    const int grid = tiles < num_sms ? tiles : num_sms;
    return launch_tc<DENSE>(ta, ta, tb, p, grid, s, "gemm_bf16");
}

cudaError_t launch_grouped(const GroupedArgs& g, cudaStream_t s) {
    const int P = g.T * g.k;
    int4* units = reinterpret_cast<int4*>(g.tiles);
    const int cap = g.tiles_cap - 1;
    cudaError_t e;
    gather_rows_kernel<<<(P + 7) / 8, 256, 0, s>>>(g.x, g.perm, P, g.k, g.d, g.xp, g.xp_exp, g.h_amax);
    trace_mark("gather_rows", s);
    build_units_kernel<<<1, 256, 0, s>>>(g.counts, g.offsets, g.E, kUnitRows, units, cap);
    trace_mark("build_units", s);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;

    // UP: A = w1 / w3 raw bytes [E*f, d/2], B = xp [P, d] f16
    CUtensorMap t1, t3, tb;
    const uint64_t rows_up = static_cast<uint64_t>(g.E) * g.f;
    if (!make_tmap(&t1, g.w1_q, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, g.d / 2, rows_up, BK / 2, BM,
                   CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_tmap(&t3, g.w3_q, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, g.d / 2, rows_up, BK / 2, BM,
                   CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_tmap(&tb, g.xp, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, g.d, P, BK, kUnitRows,
                   CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorNotSupported;
    TcParams p{};
    p.K = g.d;
    p.rows_per_expert = g.f;
    p.m_tiles = (g.f + BM - 1) / BM;
    p.s1 = g.w1_s;
    p.s3 = g.w3_s;
    p.units = units;
    p.bexp = g.xp_exp;
    p.n_out = g.f;
    p.hf = g.hf;
    p.h_amax = g.h_amax;
    p.hdr = g.hdr;
    if ((e = launch_tc<UP>(t1, t3, tb, p, g.num_sms, s, "expert_up")) != cudaSuccess) return e;

    convert_h_kernel<<<(P + 7) / 8, 256, 0, s>>>(g.hf, g.h_amax, P, g.f, g.hp, g.hp_exp);
    trace_mark("convert_h", s);

    // DOWN: A = w2 raw bytes [E*d, f/2], B = hp [P, f] f16
    CUtensorMap t2, th;
    const uint64_t rows_dn = static_cast<uint64_t>(g.E) * g.d;
    if (!make_tmap(&t2, g.w2_q, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, g.f / 2, rows_dn, BK / 2, BM,
                   CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_tmap(&th, g.hp, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, g.f, P, BK, kUnitRows,
                   CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorNotSupported;
    TcParams q{};
    q.K = g.f;
    q.rows_per_expert = g.d;
    q.m_tiles = (g.d + BM - 1) / BM;
    q.s1 = g.w2_s;
    q.units = units;
    q.bexp = g.hp_exp;
    q.n_out = g.d;
    q.y = g.y;
    q.hdr = g.hdr;
    if ((e = launch_tc<DOWN>(t2, t2, th, q, g.num_sms, s, "expert_down")) != cudaSuccess) return e;

    return launch_combine(g.y, 1, g.wts, g.inv, g.T, g.k, g.d, g.out, s);
}

}  // namespace k3
