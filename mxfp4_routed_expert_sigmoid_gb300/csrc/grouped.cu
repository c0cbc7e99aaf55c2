// tcgen05 GEMMs: the grouped expert GEMMs of the routed layer and the dense
// bf16 GEMM used for the latent projections and the router at large T.
//
// Two persistent, warp-specialised kernels compute
//     D[m, n] = sum_c A[m, c] * B[n, c]       (A: weights, B: token rows)
// with M = 128 weight rows per tile (TMEM lanes), N = up to BN token rows
// per tile (TMEM columns, fp32), K in stages of 64 (128 bytes of f16/bf16
// per row: the 128-byte swizzled K-major shared-memory layout of tcgen05):
// tc_dense_kernel (bf16 operands, both by TMA) and tc_expert_kernel (MXFP4
// weights dequantised to f16 in shared memory, f16 token rows by TMA).
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

#include <algorithm>
#include <atomic>
#include <mutex>

#include "common.cuh"
#include "tc.cuh"

namespace k3 {
namespace {

using namespace tc;

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int kTileA = BM * BK * 2;   // 16 KB of f16/bf16

// ---------------------------------------------------------------------------
// Dense bf16 GEMM: out[t, n] = sum_c x[t, c] * w[n, c]
//
// A = w (128 output rows per tile, TMEM lanes), B = x (256 token rows per
// tile, TMEM columns), both by TMA with 128-byte swizzle, 4 stages of 48 KB.
// Warp 0 producer, warp 1 MMA issuer, warp 2 TMEM owner, warps 4..7
// epilogue (bf16 or fp32 stores, coalesced along the output features).
// ---------------------------------------------------------------------------
struct DenseParams {
    int K;        // reduction length (multiple of 64)
    int m_tiles;  // 128-row tiles over N_out
    int T;        // token rows
    int n_tiles;  // token tiles
    void* out;    // [T, N_out] bf16 or fp32
    int out_fp32;
    int n_out;
    WsHeader* hdr;
    uint64_t* st;  // stamp slot (null: off)
};

constexpr int kDenseBN = 256, kDenseStages = 4, kDenseThreads = 256, kDenseTmemCols = 512;

constexpr size_t dense_smem_bytes() {
    return 1024 + static_cast<size_t>(kDenseStages) * (kTileA + kDenseBN * BK * 2) + 256;
}

__device__ __forceinline__ float silu_f32(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

// Per-token maxima over a warp: a[i] holds lane l's value for token i (16
// tokens).  Each step trades half of the values with the partner lane
// (offsets 16, 8, 4, 2), keeping the maxima of the half whose tokens this
// lane keeps, then a last exchange with lane ^ 1; 16 shuffles in all instead
// of 5 per token.  Returns the token whose warp maximum a[0] now holds (lanes
// l and l ^ 1 hold the same token).
__device__ __forceinline__ int token_max16(float (&a)[16], int lane) {
#pragma unroll
    for (int w = 8; w >= 1; w >>= 1) {
        const bool hi = (lane & (2 * w)) != 0;
#pragma unroll
        for (int j = 0; j < w; ++j) {
            const float send = hi ? a[j] : a[j + w];
            const float keep = hi ? a[j + w] : a[j];
            a[j] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, 2 * w));
        }
    }
    a[0] = fmaxf(a[0], __shfl_xor_sync(0xffffffffu, a[0], 1));
    return ((lane >> 4) & 1) * 8 + ((lane >> 3) & 1) * 4 + ((lane >> 2) & 1) * 2 + ((lane >> 1) & 1);
}

// Prepared scale atoms: per expert ceil(rows / 128) tiles of G = ceil(K / 128)
// atoms (zero-padded); row r of expert e is row m = r % 128 of atom tile
// e * tiles_e + r / 128, its block b at byte (b / 4) * 512 + 16 (m % 32) +
// 4 (m / 32) + b % 4 of the tile's atoms.

// Largest E8M0 exponent of the four rows m0 + 32 k (k = 0..3) of a 128-row
// tile from its prepared atoms: in every 512-byte atom, bytes 16 m0 .. 16 m0
// + 15 are those rows' four blocks (word k = row m0 + 32 k), so one 16-byte
// load per atom serves all four; the loads go out eight atoms at a time.
__device__ __forceinline__ void rows_emax_sf(const uint8_t* atoms, int G, int m0, int (&em)[4]) {
    uint32_t mx[4] = {0u, 0u, 0u, 0u};
    const uint8_t* base = atoms + 16 * m0;
    for (int s0 = 0; s0 < G; s0 += 8) {
        uint4 v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            v[i] = s0 + i < G ? ldg_nc_v4(base + static_cast<size_t>(s0 + i) * 512) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            mx[0] = __vmaxu4(mx[0], v[i].x);
            mx[1] = __vmaxu4(mx[1], v[i].y);
            mx[2] = __vmaxu4(mx[2], v[i].z);
            mx[3] = __vmaxu4(mx[3], v[i].w);
        }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k)
        em[k] = static_cast<int>(max(max(mx[k] & 0xFF, (mx[k] >> 8) & 0xFF), max((mx[k] >> 16) & 0xFF, mx[k] >> 24)));
}

// largest exponent of a canonical E8M0 row (nv 16-byte vectors), the loads
// issued four at a time
__device__ __forceinline__ int row_emax_canon(const uint8_t* row, int nv) {
    uint32_t m = 0;
    for (int i0 = 0; i0 < nv; i0 += 4) {
        uint4 v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            v[i] = i0 + i < nv ? ldg_nc_v4(row + 16 * (i0 + i)) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int i = 0; i < 4; ++i) m = __vmaxu4(m, __vmaxu4(__vmaxu4(v[i].x, v[i].y), __vmaxu4(v[i].z, v[i].w)));
    }
    return static_cast<int>(max(max(m & 0xFF, (m >> 8) & 0xFF), max((m >> 16) & 0xFF, m >> 24)));
}

// byte i (0..15) of a 16-byte vector
__device__ __forceinline__ int vec_byte(const uint4& v, int i) {
    const uint32_t w = i < 8 ? (i < 4 ? v.x : v.y) : (i < 12 ? v.z : v.w);
    return static_cast<int>((w >> (8 * (i & 3))) & 0xFF);
}

__global__ void __launch_bounds__(kDenseThreads, 1)
tc_dense_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                DenseParams p) {
    constexpr int BN = kDenseBN, STAGES = kDenseStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;                     // [STAGES][16 KB]
    uint8_t* sB = sA + STAGES * kTileA;     // [STAGES][BN * 128]
    uint64_t* full = reinterpret_cast<uint64_t*>(sB + STAGES * BN * BK * 2);
    uint64_t* empty = full + STAGES;
    uint64_t* acc_full = empty + STAGES;    // [2]
    uint64_t* acc_empty = acc_full + 2;     // [2]
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(acc_empty + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_tiles = p.n_tiles * p.m_tiles;
    stamp_start(p.st);
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
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
                     "r"(kDenseTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
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
            for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
                const int mt = tile % p.m_tiles, row0 = (tile / p.m_tiles) * BN;
                bool ok = true;
                for (int ks = 0; ks < k_stages; ++ks) {
                    if (!mbar_wait(&empty[s], ph ^ 1, abort_flag, p.hdr, 10)) { ok = false; break; }
                    mbar_expect_tx(&full[s], kTileA + BN * BK * 2);
                    tma_load_2d(sA + s * kTileA, &tmA, &full[s], ks * BK, mt * BM);
                    tma_load_2d(sB + s * BN * BK * 2, &tmB, &full[s], ks * BK, row0);
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
            const uint32_t idesc = idesc_f16(1, BM, BN);
            for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++it) {
                const int acc = it & 1;
                const uint32_t acc_ph = (it >> 1) & 1;
                if (!mbar_wait(&acc_empty[acc], acc_ph ^ 1, abort_flag, p.hdr, 20)) break;
                tc_fence_after();
                const uint32_t d0 = tmem_base + static_cast<uint32_t>(acc * BN);
                bool ok = true;
                for (int ks = 0; ks < k_stages; ++ks) {
                    if (!mbar_wait(&full[s], ph, abort_flag, p.hdr, 21)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(sA + s * kTileA);
                    const uint32_t b_addr = smem_u32(sB + s * BN * BK * 2);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        mma_f16(d0, sw128_desc(a_addr + kk * 32), sw128_desc(b_addr + kk * 32), idesc,
                                (ks > 0 || kk > 0) ? 1u : 0u);
                    mma_commit(&empty[s]);
                    if (++s == STAGES) { s = 0; ph ^= 1; }
                }
                if (!ok) break;
                mma_commit(&acc_full[acc]);
            }
        }
    } else if (warp >= 4) {
        // ------------------------------ epilogue ------------------------------
        const int wr = warp & 3;
        const int m = wr * 32 + lane;  // accumulator lane = output feature in the tile
        int it = 0;
        for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++it) {
            const int mt = tile % p.m_tiles, row0 = (tile / p.m_tiles) * BN;
            const int nrows = min(BN, p.T - row0);
            const int acc = it & 1;
            const uint32_t acc_ph = (it >> 1) & 1;
            if (!__all_sync(0xffffffffu, mbar_wait(&acc_full[acc], acc_ph, abort_flag, p.hdr, 30)))
                break;
            tc_fence_after();
            const uint32_t tbase = tmem_base + (static_cast<uint32_t>(wr * 32) << 16) +
                                   static_cast<uint32_t>(acc * BN);
            const int col = mt * BM + m;
            for (int n0 = 0; n0 < BN; n0 += 16) {
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
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[acc]);
        }
    }

    tc_fence_before();
    __syncthreads();
    stamp_end(p.st);
    if (warp == 2) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                     "r"(kDenseTmemCols));
    }
}

// ---------------------------------------------------------------------------
// Expert GEMM kernel (UP: NA = 2 matrices w1/w3, DOWN: NA = 1 matrix w2)
//
// Warps: 0 raw-weight producer (TMA into an RE-deep ring of packed E2M1
// entries, each 128 rows x 256 inputs: four 64-input stages, one 128-byte
// box row per weight row), 1 and 16 MMA issuers, 2 TMEM owner and exponent
// helper (computes each tile's per-row E8M0 maximum e_ref ahead of time into
// a small ring), 3 token producer (one TMA box of BN token rows per stage
// into a BS-deep ring; in a tile of fewer rows the rest of the box is rows
// of the next expert or zero fill, which the MMAs never read: one copy per
// stage costs less than several smaller ones), 4..7 and 17..24 epilogue
// (three sets, one warp per TMEM lane quadrant in each, taking 16-token
// chunks in turn), 8..15 dequantisation (raw ring -> f16 A stages of an
// AS-deep ring in TMEM).
//
// What bounds it, measured on this part: a thread needs about 60 ns (100 ns
// when its SM sub-partition is also running dequantising warps) to issue one
// tcgen05.mma, whatever its N, so the tiles take as many tokens per MMA as
// the tensor memory allows, and two issuers share each stage: in the up
// projection issuer i takes matrix i (w1 or w3, its own accumulator), in the
// down projection issuer i takes token columns [96 i, 96 i + 96) of the
// 192-wide accumulator, so the epilogue reads the same layout either way.
// The f16 weights never touch shared memory: each dequantising thread writes
// its row's 32 values of a stage straight into tensor memory (tcgen05.st,
// lane = weight row), and the MMAs read A from there (the A-in-TMEM form of
// tcgen05.mma), so shared memory carries only the raw codes and the token
// rows.  Three rings with their own full/empty barriers: the raw weights and
// the token rows are fetched several stages ahead (HBM and L2 latency), while
// the f16 stages only have to cover the dequantise -> MMA hand-off.
// ---------------------------------------------------------------------------
template <int NA>
struct ExpCfg;
// RE: raw-weight entries (four stages each), AS: dequantised A groups (in
// TMEM), BS: token (B) groups, NBUF: accumulator buffers in TMEM, SUB:
// 64-input stages per group, handed over together (one set of barrier waits,
// arrivals and commits per group).  TMEM (512 columns of 128 lanes) holds NBUF
// x NA accumulators of BN fp32 columns, then AS x NA x SUB A stages of 32
// columns (64 f16 inputs per row).  The up projection takes 192 token rows
// per tile with one accumulator buffer (2 x 192 + 2 x 2 x 32 = 512): its
// epilogue does not overlap the next tile's MMAs, which costs less than
// issuing twice as many 96-wide MMAs would.  The down projection takes 192
// rows with two buffers (2 x 192 + 2 x 2 x 32 = 512), so its epilogue runs
// under the next tile's MMAs.  Every hand-off costs the dequantising warps
// and the issuers a fixed time, so the down projection, whose TMEM has room
// for two-stage A groups, takes its stages in pairs; the up projection's A
// ring (two single stages) cannot grow without losing the dequantise / MMA
// overlap.
template <>
struct ExpCfg<2> {
    static constexpr int BN = 192, RE = 3, AS = 2, BS = 4, NBUF = 1, SUB = 1, TMEM_COLS = 512;
};
template <>
struct ExpCfg<1> {
    static constexpr int BN = 192, RE = 4, AS = 2, BS = 3, NBUF = 2, SUB = 2, TMEM_COLS = 512;
};
template <int NA>
constexpr int exp_acol() { return ExpCfg<NA>::NBUF * NA * ExpCfg<NA>::BN; }  // first A column
static_assert(exp_acol<2>() + ExpCfg<2>::AS * 2 * ExpCfg<2>::SUB * 32 <= 512, "up: TMEM budget");
static_assert(exp_acol<1>() + ExpCfg<1>::AS * 1 * ExpCfg<1>::SUB * 32 <= 512, "down: TMEM budget");
constexpr int kES = 4;          // exponent-reference slots (tiles ahead)
constexpr int kBoxRows = 16;    // token-row granule of the MMAs' N
constexpr int kSub = 4;         // 64-input stages per raw-weight entry
constexpr int kRawEntry = BM * kSub * BK / 2;  // 16 KB of packed E2M1: 128 rows x 128 bytes
constexpr int kSfEntry = kSub / 2 * 512;       // the entry's two prepared scale atoms
static_assert(kSub % ExpCfg<1>::SUB == 0 && kSub % ExpCfg<2>::SUB == 0, "a hand-off group ends at most one entry");
constexpr int kEpiSets = 3;       // epilogue warp sets (4 warps each: 4..7, then 17.. in fours)
constexpr int kExpThreads = 32 * (17 + 4 * (kEpiSets - 1));  // 16 is the second MMA issuer
constexpr int kDownHalf = 96;     // token columns per issuer in the down projection
static_assert(ExpCfg<1>::BN == 2 * kDownHalf, "down: two issuers split the tile's token columns");

struct ExpParams {
    int K;                // reduction length (multiple of 64)
    int rows_per_expert;  // rows of one expert matrix (multiple of 64)
    int tiles_e;          // 128-row tiles per expert (the last may be partial)
    int G;                // 128-wide scale groups per row (prepared atoms)
    const uint8_t* s1;    // E8M0 scales of A (w1 or w2): prepared atoms, or canonical rows (SFC)
    const uint8_t* s3;    // UP: the same for w3
    const int4* tiles;    // tiles[0].x = count; tiles[1 + i] = (e, first B row, B rows, m tile)
    const int32_t* bexp;  // per B row power-of-two exponent
    int n_out;            // row length of hf / y
    float* hf;            // UP: h in fp32 [P, f]
    uint32_t* h_amax;     // UP: max |h| per row (fp32 bits)
    float* y;             // DOWN: [P, d]
    WsHeader* hdr;
    uint64_t* st;         // stamp slot (null: off)
};

template <int NA>
constexpr size_t exp_smem_bytes() {
    using C = ExpCfg<NA>;
    size_t b = 1024;
    b += static_cast<size_t>(C::BS) * C::SUB * C::BN * BK * 2;
    b += static_cast<size_t>(C::RE) * NA * (kRawEntry + kSfEntry);
    b += static_cast<size_t>(kES) * NA * BM * 4;
    b += 512;
    return b;
}

// SFC = 0: the scales are prepared atoms, two 512-byte atoms per entry copied
// with the raw codes; SFC = 1: canonical E8M0 rows (K a multiple of 512), read
// by each dequantising thread straight from global memory, 16 blocks (eight
// stages) per 16-byte load, the next load issued eight stages ahead.
template <int NA, int SFC>
__global__ void __launch_bounds__(kExpThreads, 1)
tc_expert_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA3,
                 const __grid_constant__ CUtensorMap tmB, ExpParams p) {
    using C = ExpCfg<NA>;
    constexpr int BN = C::BN, RE = C::RE, AS = C::AS, BS = C::BS, SUB = C::SUB;
    constexpr int kBStage = BN * BK * 2;  // one 64-input stage of token rows
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sB = smem;                                // [BS][BN * 128]
    uint8_t* sRaw = sB + BS * SUB * kBStage;           // [RE][NA][16 KB], 128-byte swizzle
    uint8_t* sRawSf = sRaw + RE * NA * kRawEntry;      // [RE][NA][1 KB]: the entry's scale atoms
    int* sE = reinterpret_cast<int*>(sRawSf + RE * NA * kSfEntry);  // [kES][NA][128]
    uint64_t* raw_full = reinterpret_cast<uint64_t*>(sE + kES * NA * BM);
    uint64_t* raw_empty = raw_full + RE;
    uint64_t* b_full = raw_empty + RE;
    uint64_t* b_empty = b_full + BS;
    uint64_t* a_full = b_empty + BS;
    uint64_t* a_empty = a_full + AS;
    uint64_t* acc_full = a_empty + AS;
    uint64_t* acc_empty = acc_full + 2;
    uint64_t* eref_full = acc_empty + 2;
    uint64_t* eref_empty = eref_full + kES;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(eref_empty + kES);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_tiles = p.tiles[0].x;
    const int k_stages = p.K / BK;
    const int k_entries = (k_stages + kSub - 1) / kSub;
    const int k_groups = (k_stages + SUB - 1) / SUB;  // hand-off groups per tile
    stamp_start(p.st);

    if (threadIdx.x == 0) {
        for (int i = 0; i < RE; ++i) {
            mbar_init(&raw_full[i], 1);
            mbar_init(&raw_empty[i], 8);
        }
        for (int i = 0; i < BS; ++i) {
            mbar_init(&b_full[i], 1);
            mbar_init(&b_empty[i], 2);  // both issuers
        }
        for (int i = 0; i < AS; ++i) {
            mbar_init(&a_full[i], 8);
            mbar_init(&a_empty[i], 2);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&acc_full[i], 2);
            mbar_init(&acc_empty[i], 4 * kEpiSets);  // every epilogue warp
        }
        for (int i = 0; i < kES; ++i) {
            mbar_init(&eref_full[i], 1);
            mbar_init(&eref_empty[i], 4 * kEpiSets + 8);  // epilogue + dequantising warps
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
        if (NA == 2) prefetch_tmap(&tmA3);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    if (warp == 0) {
        // ---------------------------- raw-weight producer --------------------
        if (lane == 0) {
            int r = 0;
            uint32_t ph = 0;
            for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
                const int4 tl = p.tiles[1 + tile];
                const int arow = tl.x * p.rows_per_expert + tl.w * BM;
                // the tile's prepared scale atoms, one per 128 inputs (two stages)
                const size_t atoms = static_cast<size_t>(tl.x * p.tiles_e + tl.w) * p.G * 512;
                bool ok = true;
                for (int en = 0; en < k_entries; ++en) {
                    if (!mbar_wait(&raw_empty[r], ph ^ 1, abort_flag, p.hdr, 50)) { ok = false; break; }
                    // a last entry of fewer stages: the box past the row end is
                    // zero-filled (and counted); only its own atoms are copied
                    const int nst = min(kSub, k_stages - en * kSub);
                    const int sfb = SFC ? 0 : (nst + 1) / 2 * 512;
                    mbar_expect_tx(&raw_full[r], NA * (kRawEntry + sfb));
                    const size_t atom = atoms + static_cast<size_t>(en * kSub / 2) * 512;
                    tma_load_2d(sRaw + (r * NA) * kRawEntry, &tmA, &raw_full[r], en * kSub * BK / 2, arow);
                    if (!SFC) bulk_load(sRawSf + (r * NA) * kSfEntry, p.s1 + atom, sfb, &raw_full[r]);
                    if (NA == 2) {
                        tma_load_2d(sRaw + (r * NA + 1) * kRawEntry, &tmA3, &raw_full[r], en * kSub * BK / 2, arow);
                        if (!SFC) bulk_load(sRawSf + (r * NA + 1) * kSfEntry, p.s3 + atom, sfb, &raw_full[r]);
                    }
                    if (++r == RE) { r = 0; ph ^= 1; }
                }
                if (!ok) break;
            }
        }
    } else if (warp == 3) {
        // ---------------------------- token producer -------------------------
        if (lane == 0) {
            int b = 0;
            uint32_t ph = 0;
            for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
                const int4 tl = p.tiles[1 + tile];
                bool ok = true;
                for (int gs = 0; gs < k_groups; ++gs) {
                    if (!mbar_wait(&b_empty[b], ph ^ 1, abort_flag, p.hdr, 51)) { ok = false; break; }
                    const int nsub = min(SUB, k_stages - gs * SUB);
                    mbar_expect_tx(&b_full[b], nsub * kBStage);
                    for (int j = 0; j < nsub; ++j)
                        tma_load_2d(sB + (b * SUB + j) * kBStage, &tmB, &b_full[b], (gs * SUB + j) * BK, tl.y);
                    if (++b == BS) { b = 0; ph ^= 1; }
                }
                if (!ok) break;
            }
        }
    } else if (warp == 1 || warp == 16) {
        // ---------------------------- MMA issuers ----------------------------
        if (lane == 0) {
            const int me = warp == 16;
            int a = 0, b = 0;
            uint32_t aph = 0, bph = 0;
            int it = 0;
            for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++it) {
                const int4 tl = p.tiles[1 + tile];
                const int acc = C::NBUF == 2 ? (it & 1) : 0;
                const uint32_t acc_ph = C::NBUF == 2 ? ((it >> 1) & 1) : (it & 1);
                const int n_mma = ((tl.z + kBoxRows - 1) / kBoxRows) * kBoxRows;
                // up: matrix `me`, all token columns; down: token columns
                // [96 me, 96 me + n_me), possibly none
                const int m_me = NA == 2 ? me : 0;
                const int c_me = NA == 2 ? me * BN : me * kDownHalf;
                const int n_me = NA == 2 ? n_mma : (me ? max(0, n_mma - kDownHalf) : min(n_mma, kDownHalf));
                const uint32_t idesc = idesc_f16(0, BM, n_me > 0 ? n_me : 16);
                if (!mbar_wait(&acc_empty[acc], acc_ph ^ 1, abort_flag, p.hdr, 52)) break;
                tc_fence_after();
                const uint32_t d0 = tmem_base + static_cast<uint32_t>(acc * NA * BN + c_me);
                bool ok = true;
                for (int gs = 0; gs < k_groups; ++gs) {
                    if (!mbar_wait(&b_full[b], bph, abort_flag, p.hdr, 53) ||
                        !mbar_wait(&a_full[a], aph, abort_flag, p.hdr, 54)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (n_me > 0) {
                        const int nsub = min(SUB, k_stages - gs * SUB);
                        for (int j = 0; j < nsub; ++j) {
                            const uint32_t b_addr =
                                smem_u32(sB + (b * SUB + j) * kBStage + (NA == 2 ? 0 : c_me) * BK * 2);
                            // A stage (a, m_me, j): TMEM columns, 8 per 16-wide K slice
                            const uint32_t a_tm = tmem_base + static_cast<uint32_t>(
                                                                  exp_acol<NA>() + ((a * NA + m_me) * SUB + j) * 32);
#pragma unroll
                            for (int kk = 0; kk < BK / 16; ++kk)
                                mma_f16_ts(d0, a_tm + 8 * kk, sw128_desc(b_addr + kk * 32), idesc,
                                           (gs > 0 || j > 0 || kk > 0) ? 1u : 0u);
                        }
                        mma_commit(&a_empty[a]);
                        mma_commit(&b_empty[b]);
                    } else {
                        mbar_arrive(&a_empty[a]);
                        mbar_arrive(&b_empty[b]);
                    }
                    if (++a == AS) { a = 0; aph ^= 1; }
                    if (++b == BS) { b = 0; bph ^= 1; }
                }
                if (!ok) break;
                if (n_me > 0)
                    mma_commit(&acc_full[acc]);
                else
                    mbar_arrive(&acc_full[acc]);
            }
        }
    } else if (warp == 2) {
        // ---------------------------- exponent helper ------------------------
        int it = 0;
        for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++it) {
            const int4 tl = p.tiles[1 + tile];
            const int slot = it % kES;
            const uint32_t eph = (it / kES) & 1;
            if (!__all_sync(0xffffffffu, mbar_wait(&eref_empty[slot], eph ^ 1, abort_flag, p.hdr, 55)))
                break;
#pragma unroll
            for (int m = 0; m < NA; ++m) {
                const uint8_t* sm_ = m == 0 ? p.s1 : p.s3;
                int em[4];
                if (SFC) {
                    // rows lane + 32 k of the tile; a row past the expert gets 0
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int r = tl.w * BM + lane + 32 * k;
                        em[k] = r < p.rows_per_expert
                                    ? row_emax_canon(sm_ + (static_cast<size_t>(tl.x) * p.rows_per_expert + r) *
                                                               (p.K / 32),
                                                     p.K / 512)
                                    : 0;
                    }
                } else {
                    // a partial last tile's atoms are zero-padded: its missing rows read 0
                    rows_emax_sf(sm_ + static_cast<size_t>(tl.x * p.tiles_e + tl.w) * p.G * 512, p.G, lane, em);
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) sE[(slot * NA + m) * BM + lane + 32 * k] = em[k];
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&eref_full[slot]);
        }
    } else if ((warp >= 4 && warp < 8) || warp >= 17) {
        // ---------------------------- epilogue -------------------------------
        // kEpiSets sets of four warps (4..7, then 17.. in fours), one warp per
        // TMEM lane quadrant in each; set h takes the 16-token chunks
        // kEpiSets j + h
        const int wr = warp & 3;
        const int eset = warp >= 17 ? 1 + (warp - 17) / 4 : 0;
        const int m = wr * 32 + lane;
        int it = 0;
        for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++it) {
            const int4 tl = p.tiles[1 + tile];
            const int acc = C::NBUF == 2 ? (it & 1) : 0;
            const uint32_t acc_ph = C::NBUF == 2 ? ((it >> 1) & 1) : (it & 1);
            const int slot = it % kES;
            const uint32_t eph = (it / kES) & 1;
            if (!__all_sync(0xffffffffu, mbar_wait(&acc_full[acc], acc_ph, abort_flag, p.hdr, 56) &&
                                             mbar_wait(&eref_full[slot], eph, abort_flag, p.hdr, 57)))
                break;
            tc_fence_after();
            const uint32_t tbase = tmem_base + (static_cast<uint32_t>(wr * 32) << 16) +
                                   static_cast<uint32_t>(acc * NA * BN);
            const int nrows = tl.z, row0 = tl.y;
            const int n_used = ((nrows + kBoxRows - 1) / kBoxRows) * kBoxRows;
            const int r = tl.w * BM + m;
            const bool valid = r < p.rows_per_expert;
            const int eref1 = sE[(slot * NA + 0) * BM + m];
            const int eref3 = NA == 2 ? sE[(slot * NA + (NA - 1)) * BM + m] : 0;
            for (int n0 = 16 * eset; n0 < n_used; n0 += 16 * kEpiSets) {
                // tokens n0 .. n0 + cnt - 1 of the tile are real; lane i < cnt
                // fetches token i's exponent for the whole warp
                const int cnt = min(16, nrows - n0);
                const int xe_l = lane < cnt ? p.bexp[row0 + n0 + lane] : 0;
                if (NA == 2) {
                    float v1[16], v3[16], a[16];
                    tmem_ld16x2(tbase + n0, tbase + BN + n0, v1, v3);
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int xe = __shfl_sync(0xffffffffu, xe_l, i);
                        const float gg = mul_pow2(v1[i], eref1 - 127 + xe);
                        const float u = mul_pow2(v3[i], eref3 - 127 + xe);
                        const float h = silu_f32(gg) * u;
                        if (valid && i < cnt) p.hf[static_cast<size_t>(row0 + n0 + i) * p.n_out + r] = h;
                        a[i] = valid ? fabsf(h) : 0.0f;
                    }
                    const int t = token_max16(a, lane);
                    if ((lane & 1) == 0 && t < cnt) atomicMax(p.h_amax + row0 + n0 + t, __float_as_uint(a[0]));
                } else {
                    float v1[16];
                    tmem_ld16(tbase + n0, v1);
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int xe = __shfl_sync(0xffffffffu, xe_l, i);
                        const float yv = mul_pow2(v1[i], eref1 - 127 + xe);
                        if (valid && i < cnt) p.y[static_cast<size_t>(row0 + n0 + i) * p.n_out + r] = yv;
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&acc_empty[acc]);
                mbar_arrive(&eref_empty[slot]);
            }
        }
    } else if (warp >= 8 && warp < 16) {
        // ---------------------------- dequantisation -------------------------
        // warp 8 + 4 half + q: TMEM lane quadrant q, one weight row per lane,
        // inputs 32 half .. 32 half + 31 of each 64-wide stage
        const int q = warp & 3, half = (warp - 8) >> 2;
        const int row = 32 * q + lane;
        const uint32_t a_lane = tmem_base + (static_cast<uint32_t>(32 * q) << 16) +
                                static_cast<uint32_t>(exp_acol<NA>() + 16 * half);
        int r = 0, a = 0;
        uint32_t rph = 0, aph = 0;
        int it = 0;
        const int swz = row & 7;  // 128-byte swizzle of the raw entries: 16-byte chunk j sits at j ^ (row % 8)
        for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++it) {
            const int4 tl = p.tiles[1 + tile];
            const int slot = it % kES;
            const uint32_t eph = (it / kES) & 1;
            if (!__all_sync(0xffffffffu, mbar_wait(&eref_full[slot], eph, abort_flag, p.hdr, 58))) break;
            const int eref1 = sE[(slot * NA + 0) * BM + row];
            const int eref3 = NA == 2 ? sE[(slot * NA + (NA - 1)) * BM + row] : 0;
            // this thread's byte of a scale atom: row `row`, block 2 ks + half
            // (an entry holds two atoms: stages 0-1 and 2-3)
            const int sfo = 16 * (row & 31) + 4 * (row >> 5);
            // canonical scales: the row's 16-byte vectors, current and next (a
            // row past the expert reads zeros: its products are never stored)
            const int grow = tl.w * BM + row;
            const bool rvalid = grow < p.rows_per_expert;
            const int nvec = p.K / 512;
            const uint8_t* c1 = p.s1 + (static_cast<size_t>(tl.x) * p.rows_per_expert + grow) * (p.K / 32);
            const uint8_t* c3 = NA == 2 ? p.s3 + (c1 - p.s1) : nullptr;
            uint4 v1 = make_uint4(0, 0, 0, 0), v3 = v1, n1 = v1, n3 = v1;
            if (SFC && rvalid) {
                n1 = ldg_nc_v4(c1);
                if (NA == 2) n3 = ldg_nc_v4(c3);
            }
            bool ok = true;
            for (int gs = 0; gs < k_groups; ++gs) {
                const int nsub = min(SUB, k_stages - gs * SUB);
                if (!__all_sync(0xffffffffu, mbar_wait(&a_empty[a], aph ^ 1, abort_flag, p.hdr, 60))) {
                    ok = false;
                    break;
                }
                tc_fence_after();  // the MMAs that read this A group have completed
                int ended = -1;    // the raw entry whose last stage is in this group
                for (int j = 0; j < nsub; ++j) {
                    const int ks = gs * SUB + j;
                    const int blk = 2 * ks + half;
                    if (SFC && (ks & 7) == 0) {
                        v1 = n1;
                        v3 = n3;
                        if (rvalid && (ks >> 3) + 1 < nvec) {
                            n1 = ldg_nc_v4(c1 + 16 * ((ks >> 3) + 1));
                            if (NA == 2) n3 = ldg_nc_v4(c3 + 16 * ((ks >> 3) + 1));
                        }
                    }
                    const int sub = ks % kSub;  // stage within the raw entry
                    if (sub == 0 &&
                        !__all_sync(0xffffffffu, mbar_wait(&raw_full[r], rph, abort_flag, p.hdr, 59))) {
                        ok = false;
                        break;
                    }
                    int e1, e3;
                    if (SFC) {
                        e1 = vec_byte(v1, blk & 15);
                        e3 = NA == 2 ? vec_byte(v3, blk & 15) : 0;
                    } else {
                        const int sfb = (sub >> 1) * 512 + sfo + (blk & 3);
                        e1 = sRawSf[(r * NA) * kSfEntry + sfb];
                        e3 = NA == 2 ? sRawSf[(r * NA + (NA - 1)) * kSfEntry + sfb] : 0;
                    }
#pragma unroll
                    for (int mm = 0; mm < NA; ++mm) {
                        const uint4 raw = *reinterpret_cast<const uint4*>(
                            sRaw + (r * NA + mm) * kRawEntry + row * 128 + (((2 * sub + half) ^ swz) << 4));
                        const uint16_t sh = f16_pow2(mm == 0 ? e1 - eref1 : e3 - eref3);
                        const uint32_t sc2 = static_cast<uint32_t>(sh) | (static_cast<uint32_t>(sh) << 16);
                        uint32_t w[16];
                        e2m1x8_to_f16x8(raw.x, w[0], w[1], w[2], w[3]);
                        e2m1x8_to_f16x8(raw.y, w[4], w[5], w[6], w[7]);
                        e2m1x8_to_f16x8(raw.z, w[8], w[9], w[10], w[11]);
                        e2m1x8_to_f16x8(raw.w, w[12], w[13], w[14], w[15]);
#pragma unroll
                        for (int i = 0; i < 16; ++i) w[i] = hmul2(w[i], sc2);
                        tmem_st16(a_lane + static_cast<uint32_t>(((a * NA + mm) * SUB + j) * 32), w);
                    }
                    if (sub == kSub - 1 || ks == k_stages - 1) {  // the entry's last stage
                        ended = r;
                        if (++r == RE) { r = 0; rph ^= 1; }
                    }
                }
                tmem_wait_st();
                if (!ok) break;
                tc_fence_before();
                if (ended >= 0) fence_proxy_async();  // the raw codes were read here; the producer's TMA rewrites them
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&a_full[a]);
                    if (ended >= 0) mbar_arrive(&raw_empty[ended]);
                }
                if (++a == AS) { a = 0; aph ^= 1; }
            }
            if (!ok) break;
            if (lane == 0) mbar_arrive(&eref_empty[slot]);
        }
    }

    tc_fence_before();
    __syncthreads();
    stamp_end(p.st);
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
                   uint32_t* __restrict__ h_amax, uint64_t* st) {
    StampScope stamp(st);
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
                 uint16_t* __restrict__ hp, int32_t* __restrict__ hexp, uint64_t* st) {
    StampScope stamp(st);
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

// Tile lists of the expert GEMMs: for every expert with tokens, its token
// rows are cut into chunks of at most bn rows, and each (m tile, chunk) pair
// is one tile.  Order: expert, then m tile, then chunk, so the chunks that
// share one weight tile are consecutive (neighbouring CTAs read the same
// weight bytes, mostly from L2).  list[0].x = count; list[1 + i] =
// (expert, first row, rows, m tile).
__global__ void __launch_bounds__(1024)
build_tiles_kernel(const int32_t* __restrict__ counts, const int32_t* __restrict__ offsets, int E,
                   int bn_up, int bn_dn, int m_up, int m_dn, int4* up, int4* dn, int cap, uint64_t* st) {
    StampScope stamp(st);
    // every CTA scans the per-expert chunk counts (E <= 1024, one per thread)
    // and writes its share of the list entries
    __shared__ int base[1024 + 1];
    __shared__ int wsum[32];
    __shared__ int total_s;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    for (int pass = 0; pass < 2; ++pass) {
        const int bn = pass == 0 ? bn_up : bn_dn;
        const int v = tid < E ? (counts[tid] + bn - 1) / bn : 0;
        int incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += t;
        }
        if (lane == 31) wsum[wid] = incl;
        __syncthreads();
        if (wid == 0) {
            const int w = lane < static_cast<int>(blockDim.x >> 5) ? wsum[lane] : 0;
            int wi = w;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int t = __shfl_up_sync(0xffffffffu, wi, o);
                if (lane >= o) wi += t;
            }
            wsum[lane] = wi - w;  // exclusive offsets of the warps
            if (lane == 31) total_s = wi;
        }
        __syncthreads();
        if (tid < E) base[tid] = wsum[wid] + incl - v;
        if (tid == 0) base[E] = total_s;
        __syncthreads();
        const int mt_n = pass == 0 ? m_up : m_dn;
        const int n = min(base[E] * mt_n, cap);
        int4* list = pass == 0 ? up : dn;
        if (blockIdx.x == 0 && tid == 0) list[0] = make_int4(n, 0, 0, 0);
        for (int i = blockIdx.x * blockDim.x + tid; i < n; i += gridDim.x * blockDim.x) {
            // expert of entry i: largest e with base[e] * mt_n <= i
            int lo = 0, hi = E - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (base[mid] * mt_n <= i) lo = mid; else hi = mid - 1;
            }
            const int e = lo;
            const int nch = base[e + 1] - base[e];
            const int local = i - base[e] * mt_n;
            const int mt = local / nch, c = local % nch;
            const int cnt = counts[e];
            list[1 + i] = make_int4(e, offsets[e] + c * bn, min(bn, cnt - c * bn), mt);
        }
        __syncthreads();  // base[] and wsum[] are rebuilt for the next pass
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
cudaError_t launch_dense(const CUtensorMap& a, const CUtensorMap& b, const DenseParams& p,
                         int grid, cudaStream_t s, const char* name) {
    constexpr size_t smem = dense_smem_bytes();
    static_assert(smem <= 232448, "shared memory budget");
    // the attribute is per device; set it once per device (not inside graph captures)
    static std::atomic<uint64_t> done{0};
    int dev = 0;
    cudaGetDevice(&dev);
    const uint64_t bit = 1ull << (dev & 63);
    if (!(done.load() & bit)) {
        cudaError_t e = cudaFuncSetAttribute(tc_dense_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        done.fetch_or(bit);
    }
    DenseParams q = p;
    q.st = trace_stamp(name);
    tc_dense_kernel<<<grid, kDenseThreads, smem, s>>>(a, b, q);
    trace_mark(name, s);
    return cudaGetLastError();
}

// token rows per tile of the up (W1, W3) and down (W2) passes
constexpr int kUpRows = ExpCfg<2>::BN, kDownRows = ExpCfg<1>::BN;
constexpr int kUnitRows = kUpRows < kDownRows ? kUpRows : kDownRows;  // bounds the tile count

template <int NA, int SFC>
cudaError_t launch_expert_sfc(const CUtensorMap& a, const CUtensorMap& a3, const CUtensorMap& b,
                              const ExpParams& p, int grid, cudaStream_t s, const char* name) {
    constexpr size_t smem = exp_smem_bytes<NA>();
    static_assert(smem <= 232448, "shared memory budget");
    static std::atomic<uint64_t> done{0};
    int dev = 0;
    cudaGetDevice(&dev);
    const uint64_t bit = 1ull << (dev & 63);
    if (!(done.load() & bit)) {
        cudaError_t e = cudaFuncSetAttribute(tc_expert_kernel<NA, SFC>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        done.fetch_or(bit);
    }
    ExpParams q = p;
    q.st = trace_stamp(name);
    tc_expert_kernel<NA, SFC><<<grid, kExpThreads, smem, s>>>(a, a3, b, q);
    trace_mark(name, s);
    return cudaGetLastError();
}

template <int NA>
cudaError_t launch_expert(int sf_canon, const CUtensorMap& a, const CUtensorMap& a3, const CUtensorMap& b,
                          const ExpParams& p, int grid, cudaStream_t s, const char* name) {
    return sf_canon ? launch_expert_sfc<NA, 1>(a, a3, b, p, grid, s, name)
                    : launch_expert_sfc<NA, 0>(a, a3, b, p, grid, s, name);
}

}  // namespace

size_t grouped_tile_cap(int T, int E, int k, int d, int f) {
    const size_t units = static_cast<size_t>(E) + (static_cast<size_t>(T) * k + kUnitRows - 1) / kUnitRows + 1;
    const size_t mt = static_cast<size_t>(std::max((f + BM - 1) / BM, (d + BM - 1) / BM));
    return units * mt;
}

cudaError_t launch_gemm_bf16(const uint16_t* x, const uint16_t* w, int T, int N, int K, void* out,
                             int out_fp32, WsHeader* hdr, int num_sms, cudaStream_t s, const char* name) {
    if (N % BM || K % BK || T < 1) return cudaErrorInvalidValue;
    CUtensorMap ta, tb;
    if (!make_tmap(&ta, w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, K, N, BK, BM,
                   CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorNotSupported;
    if (!make_tmap(&tb, x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, K, T, BK, kDenseBN,
                   CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorNotSupported;
    DenseParams p{};
    p.K = K;
    p.m_tiles = N / BM;
    p.T = T;
    p.n_tiles = (T + kDenseBN - 1) / kDenseBN;
    p.out = out;
    p.out_fp32 = out_fp32;
    p.n_out = N;
    p.hdr = hdr;
    const int tiles = p.n_tiles * p.m_tiles;
    const int grid = tiles < num_sms ? tiles : num_sms;
    return launch_dense(ta, tb, p, grid, s, name);
}

cudaError_t launch_grouped(const GroupedArgs& g, cudaStream_t s) {
    const int P = g.T * g.k;
    const int cap = g.tiles_cap;
    int4* tiles_up = reinterpret_cast<int4*>(g.tiles);
    int4* tiles_dn = tiles_up + (cap + 1);
    cudaError_t e;
    gather_rows_kernel<<<(P + 7) / 8, 256, 0, s>>>(g.x, g.perm, P, g.k, g.d, g.xp, g.xp_exp, g.h_amax,
                                                   trace_stamp("gather_rows"));
    trace_mark("gather_rows", s);
    build_tiles_kernel<<<g.num_sms, 1024, 0, s>>>(g.counts, g.offsets, g.E, kUpRows, kDownRows, (g.f + BM - 1) / BM,
                                          (g.d + BM - 1) / BM, tiles_up, tiles_dn, cap, trace_stamp("build_tiles"));
    trace_mark("build_tiles", s);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;

    // UP: A = w1 / w3 raw bytes [E*f, d/2] in 128-byte x 128-row boxes (a box
    // past the end of a row, d % 256 != 0, is zero-filled), B = xp [P, d] f16
    // in boxes of 192 rows
    CUtensorMap t1, t3, tb;
    const uint64_t rows_up = static_cast<uint64_t>(g.E) * g.f;
    if (!make_tmap(&t1, g.w1_q, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, g.d / 2, rows_up, kSub * BK / 2, BM,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tmap(&t3, g.w3_q, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, g.d / 2, rows_up, kSub * BK / 2, BM,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tmap(&tb, g.xp, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, g.d, P, BK, kUpRows,
                   CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorNotSupported;
    if (g.sf_canon && (g.d % 512 || g.f % 512)) return cudaErrorNotSupported;
    ExpParams p{};
    p.K = g.d;
    p.rows_per_expert = g.f;
    p.tiles_e = (g.f + BM - 1) / BM;
    p.G = (g.d + 127) / 128;
    p.s1 = g.w1_sf;
    p.s3 = g.w3_sf;
    p.tiles = tiles_up;
    p.bexp = g.xp_exp;
    p.n_out = g.f;
    p.hf = g.hf;
    p.h_amax = g.h_amax;
    p.hdr = g.hdr;
    if ((e = launch_expert<2>(g.sf_canon, t1, t3, tb, p, g.num_sms, s, "expert_up")) != cudaSuccess) return e;

    convert_h_kernel<<<(P + 7) / 8, 256, 0, s>>>(g.hf, g.h_amax, P, g.f, g.hp, g.hp_exp, trace_stamp("convert_h"));
    trace_mark("convert_h", s);

    // DOWN: A = w2 raw bytes [E*d, f/2], B = hp [P, f] f16 in boxes of 192 rows
    CUtensorMap t2, th;
    const uint64_t rows_dn = static_cast<uint64_t>(g.E) * g.d;
    if (!make_tmap(&t2, g.w2_q, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, g.f / 2, rows_dn, kSub * BK / 2, BM,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tmap(&th, g.hp, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, g.f, P, BK, kDownRows,
                   CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorNotSupported;
    ExpParams q{};
    q.K = g.f;
    q.rows_per_expert = g.d;
    q.tiles_e = (g.d + BM - 1) / BM;
    q.G = (g.f + 127) / 128;
    q.s1 = g.w2_sf;
    q.tiles = tiles_dn;
    q.bexp = g.hp_exp;
    q.n_out = g.d;
    q.y = g.y;
    q.hdr = g.hdr;
    if ((e = launch_expert<1>(g.sf_canon, t2, t2, th, q, g.num_sms, s, "expert_down")) != cudaSuccess) return e;

    return launch_combine(g.y, 1, g.wts, g.inv, g.T, g.k, g.d, g.out, s);
}

}  // namespace k3
