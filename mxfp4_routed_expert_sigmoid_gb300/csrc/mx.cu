// Block-scaled tensor-core path of the routed experts (decode, T <= 8), and
// the scale-factor layout it reads.
//
// The experts' MXFP4 weights reach the tensor cores as they are stored:
// tcgen05.mma kind::mxf4 multiplies packed E2M1 weight codes by packed E2M1
// activation codes and applies both operands' E8M0 block scales (one per 32
// inputs) in hardware, accumulating in fp32 in TMEM; nothing is dequantised
// in software (llama.cpp PR #26185 "model: add Kimi-K3 text model", review by
// GrEarl, section "repack_mxfp4_blocks is bit-exact": the MXFP4 format;
// section "Dry run": 896 experts, 16 used, latent width 3584, expert width
// 3072).
//
// Operands of one MMA (M = 128 weight rows, N = 16..64 token-term rows,
// K = 64), staged per 256-wide K chunk (128 bytes of codes per row, the
// 128-byte swizzled K-major layout), two chunks to a pipeline stage:
//   A  weight codes by TMA, 16 KB per chunk, as stored in global memory (a
//      chunk past the end of a row is zero-filled by the TMA unit, and MMAs
//      past the row's last 64 inputs are not issued);
//   SFA two 512-byte scale atoms per chunk, copied to TMEM by tcgen05.cp
//      32x128b.warpx4: row m is read from lane m, column m / 32; an MMA reads
//      two bytes of a column (scale id 0 for the first 64 inputs of an atom, 2
//      for the second).  The atoms come either prepared (the layout written by
//      k3moe_prepare_scales, one bulk copy per stage) or from the checkpoint's
//      canonical E8M0 rows: one TMA box of 16 bytes x 128 rows per stage,
//      which the two MMA issuer warps re-lay into atom order in shared memory
//      (32 lanes each, their own chunk) before the tcgen05.cp;
//   B  activations as kTerms E2M1 terms per token (rows kTerms t + j; see
//      quantize_terms), pre-swizzled in global memory, one bulk copy;
//   SFB their scale atoms (column n from lane n % 32, column n / 32).
// The kTerms partial products of a token are summed in fp32 by the epilogue.
// Why kind::mxf4: one tcgen05.mma with M = 128 takes about 55 ns on GB300
// whatever N up to 128 (measured), so the weight bytes an instruction covers
// set the speed limit: 4 KB with K = 64 here, twice kind::mxf8f6f4's K = 32.
//
// Up projection: W1 and W3 are separate units (128-row tiles of one matrix);
// the finish kernel pairs g = W1 x with u = W3 x.  Down projection: 128-row
// tiles of W2.
//
// Work split (stream-K): the units (active expert, matrix, row tile, stage)
// are cut into one contiguous range per CTA, every range at least one tile
// long, so a tile is shared by at most two CTAs.  The CTA that starts a tile
// writes its partial sums to slot 0 and the other to slot 1 (a CTA that owns
// the whole tile writes zeros to slot 1); consumers add slot 0 and slot 1 in
// that order, so results do not depend on timing.
//
// Kernels of one decode forward (after the router, which also writes the
// token rows as E2M1 terms): up -> finish (h = silu(g) * u from both slots,
// quantised to E2M1 terms) -> down -> combine (weights in slot order).
//
// Roles of the streaming kernel (224 threads, one CTA per SM):
//   warp 0     producer: TMA / bulk copies into a ring of stages;
//   warp 1     TMEM owner and MMA issuer of the first K chunk of each stage;
//   warp 6     MMA issuer of the second chunk (one issuing thread reaches about
//              60 % of the MMA rate of two, measured), into its own accumulator;
//   warps 2..5 epilogue: tcgen05.ld of the accumulator quadrant (warp % 4),
//              the two issuers' accumulators added in a fixed order.
// Every wait is bounded (kWaitLimitNs); on expiry the CTA records
// K3MOE_ERR_TIMEOUT, every role stops, copies in flight are waited for (with
// a limit) and TMEM is released.
#include <atomic>

#include "common.cuh"
#include "tc.cuh"

namespace k3 {
namespace {

using namespace tc;

constexpr int kMxThreads = 224;
constexpr int kGgThreads = 128;        // ggml-block variant: one converting thread per tile row
constexpr int kGgBar = 1;              // their named barrier
constexpr int kMaxStages = 8;
constexpr int kChunks = 2;             // 256-wide K chunks per stage (a stage covers K = 512)
constexpr int kChunkA = 16384;         // 128 rows x 128 bytes of packed E2M1
constexpr int kStageA = kChunks * kChunkA;
// ggml 17-byte blocks: a stage of one tile row is 16 blocks = 272 bytes, the
// tile's 128 rows 34,816 bytes = the A chunks and scale atoms they become
constexpr int kGgRowBytes = 4 * kChunks * 2 * 17;
constexpr int kGgStageBytes = 128 * kGgRowBytes;
static_assert(kGgStageBytes == kStageA + kChunks * 1024, "a ggml stage converts in place");
constexpr int kMaxN = 64;              // MMA N: kTerms * T rounded up to 16
// TMEM: accumulators (buffer a, issuer t) at (2 a + t) * kMaxN, then the scale
// slots, each on a 32-column boundary: issuer t's atoms A0, B0, A1, B1 of its
// chunk at kSfBase + 128 t + 32 g
constexpr int kSfBase = 4 * kMaxN;
static_assert(kChunks == 2, "one K chunk per MMA issuer");
static_assert(kSfBase + kChunks * 128 <= 512, "scale slots fit in TMEM");
constexpr uint32_t kTmemCols = 512;
// weight formats of the streaming kernel: compressed-tensors codes with
// prepared scale atoms, ggml 17-byte blocks, or codes with canonical E8M0 rows
constexpr int kWfAtoms = 0, kWfGgml = 1, kWfCanon = 2;
constexpr int kRawSf = 2048;           // canonical: one stage's scale rows, 128 x 16 bytes

__device__ __forceinline__ float silu_f32(float g) { return g / (1.0f + expf(-g)); }

// Instruction descriptor, kind::mxf4: A = B = E2M1 (format 1), E8M0 scales,
// K-major, M x N; sa / sb = scale id (0: blocks 0, 1 of the atom column; 2:
// blocks 2, 3).
__device__ __forceinline__ uint32_t idesc_f4(int M, int N, int sa, int sb) {
    return (static_cast<uint32_t>(sb) << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
           (1u << 23) | (static_cast<uint32_t>(M >> 4) << 24) | (static_cast<uint32_t>(sa) << 29);
}

__device__ __forceinline__ void mma_f4(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                       uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
        " tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5],"
        " p;\n}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate));
}

struct MxArgs {
    const uint8_t* sf[2];   // prepared scale atoms of the matrices (W1, W3 or W2; atoms format)
    int nmat;               // matrices per expert in this pass (2 up, 1 down)
    int early_a;            // 1: the active list is final before this grid's wait (down)
    const uint8_t* bq;      // B codes [unit][K / 256][N][128] (up: one shared unit)
    const uint8_t* bsf;     // B scale atoms [unit][K / 128][512]
    size_t bq_ustride;      // bytes per unit (0 when all units share B)
    size_t bsf_ustride;
    const int32_t* active;  // expert of each unit (decode: the active experts ascending)
    const int32_t* count;   // number of units (decode: active + E)
    const int32_t* ucnt;    // tokens of each unit (null: all T)
    const int32_t* ubase;   // unit-grouped: first unit of each expert, [E + 1] (null: decode)
    const int32_t* slot_of; // expert -> slot of the weight arrays (null: the expert itself)
    int nslots;             // slots the weight arrays hold
    int E;
    int rows;               // weight rows per expert (f up, d down), a multiple of 64
    int tiles;              // 128-row tiles per expert (the last may hold fewer rows)
    int K;                  // inputs (d up, f down), a multiple of 64
    int KC;                 // 256-wide K chunks (the last may be partial)
    int KS;                 // stages of kChunks chunks (the last one may be shorter)
    int G;                  // 128-wide scale groups per row (prepared atoms per tile)
    int N;                  // MMA N
    int T;                  // tokens
    int RS;                 // stages in the ring
    uint32_t stage_bytes;
    float* part;            // [slot][mat][umax][T][rows_out]
    int umax;
    int rows_out;           // f (up) or d (down)
    WsHeader* hdr;
    uint64_t* st;           // stamp slot (null: off)
    int inject;             // test aid: CTA 0 drops its first stage's signal; waits give up after 1 ms
};

// Position in the sequence of stages.  Decode: (unit, matrix, row tile,
// stage), the unit being the position in the active list.  Unit-grouped
// (ubase set): expert by expert, (matrix, row tile, unit of the expert,
// stage), so that the units of one expert read each weight tile back to back
// and all but the first find it in L2.
struct Cursor {
    int u, mat, tile, ks;
    int e, grp, ngrp;  // expert (decode: the unit), unit within the expert, units of the expert
    __device__ Cursor(int w, const MxArgs& p) {
        if (!p.ubase) {
            const int per_m = p.tiles * p.KS, per_u = p.nmat * per_m;
            u = w / per_u;
            int r = w - u * per_u;
            mat = r / per_m;
            r -= mat * per_m;
            tile = r / p.KS;
            ks = r - tile * p.KS;
            e = u;
            grp = 0;
            ngrp = 1;
        } else {
            const int su = p.nmat * p.tiles * p.KS;  // stages per unit
            int lo = 0, hi = p.E - 1;               // largest e with ubase[e] * su <= w
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (p.ubase[mid] * su <= w) lo = mid;
                else hi = mid - 1;
            }
            e = lo;
            ngrp = p.ubase[e + 1] - p.ubase[e];
            int r = w - p.ubase[e] * su;
            const int per_tile = ngrp * p.KS, per_m = p.tiles * per_tile;
            mat = r / per_m;
            r -= mat * per_m;
            tile = r / per_tile;
            r -= tile * per_tile;
            grp = r / p.KS;
            ks = r - grp * p.KS;
            u = p.ubase[e] + grp;
        }
    }
    // the first stage of the next (unit, matrix, row tile)
    __device__ void next_segment(const MxArgs& p) {
        ks = 0;
        if (++grp == ngrp) {
            grp = 0;
            if (++tile == p.tiles) {
                tile = 0;
                if (++mat == p.nmat) {
                    mat = 0;
                    if (p.ubase) {
                        do {
                            ++e;
                        } while (e < p.E && p.ubase[e + 1] == p.ubase[e]);
                        ngrp = e < p.E ? p.ubase[e + 1] - p.ubase[e] : 1;
                    } else {
                        ++e;
                    }
                }
            }
        }
        u = p.ubase ? (e < p.E ? p.ubase[e] : 0) + grp : e;
    }
    __device__ void next(const MxArgs& p) {
        if (++ks == p.KS) next_segment(p);
    }
};

__device__ __forceinline__ void named_bar_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// barrier over n threads that also ANDs a predicate across them
__device__ __forceinline__ bool named_bar_and(int id, int n, bool v) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, %2, %3, p;\n"
        " selp.u32 %0, 1, 0, q;\n}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(v)), "r"(id), "r"(n)
        : "memory");
    return r != 0;
}

// For a word q of ggml code bytes c_j | c_(j+16) << 4: bytes 0 and 2 of
// *lo_pairs are c_0 | c_1 << 4 and c_2 | c_3 << 4 (the word's low nibbles
// paired), bytes 0 and 2 of *hi_pairs the same for its high nibbles; bytes 1
// and 3 are left over.
__device__ __forceinline__ void nibble_pairs(uint32_t q, uint32_t* lo_pairs, uint32_t* hi_pairs) {
    constexpr uint32_t lo = 0x0F0F0F0Fu;
    const uint32_t t = q >> 4, u = q >> 8;
    *lo_pairs = (q & lo) | (t & ~lo);
    *hi_pairs = (t & lo) | (u & ~lo);
}

// One tile row of a stage stored as ggml blocks (llama.cpp PR #26185, review
// by GrEarl, "repack_mxfp4_blocks is bit-exact": 17 bytes per 32 inputs, the
// E8M0 byte unchanged, then byte j holding code j in the low and code j + 16
// in the high nibble) -> the row of the two A chunks (128-byte swizzled, code
// 2i in the low nibble of byte i, as the compressed-tensors layout stores
// them) and the row's bytes of the stage's four scale atoms.  The stage is
// converted in place: every row is read into registers before the barrier,
// then written.
__device__ __forceinline__ void gg_convert_row(uint8_t* st, int r, uint32_t offSA) {
    uint32_t R[kGgRowBytes / 4 + 1];
    const uint4* src = reinterpret_cast<const uint4*>(st + r * kGgRowBytes);
#pragma unroll
    for (int i = 0; i < kGgRowBytes / 16; ++i) {
        const uint4 v = src[i];
        R[4 * i] = v.x;
        R[4 * i + 1] = v.y;
        R[4 * i + 2] = v.z;
        R[4 * i + 3] = v.w;
    }
    R[kGgRowBytes / 4] = 0;
    named_bar_sync(kGgBar, kGgThreads);
#pragma unroll
    for (int b = 0; b < 4 * kChunks * 2; ++b) {
        const int o = 17 * b + 1, wi = o >> 2, sh = 8 * (o & 3);
        uint32_t L[4], H[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) nibble_pairs(__funnelshift_r(R[wi + i], R[wi + i + 1], sh), &L[i], &H[i]);
        uint4 n;
        n.x = __byte_perm(L[0], L[1], 0x6420);  // codes 0..7
        n.y = __byte_perm(L[2], L[3], 0x6420);  // codes 8..15
        n.z = __byte_perm(H[0], H[1], 0x6420);  // codes 16..23
        n.w = __byte_perm(H[2], H[3], 0x6420);  // codes 24..31
        const int chunk = b >> 3, unit = b & 7;
        *reinterpret_cast<uint4*>(st + chunk * kChunkA + r * 128 + ((unit ^ (r & 7)) << 4)) = n;
    }
#pragma unroll
    for (int g = 0; g < 2 * kChunks; ++g) {
        uint32_t v = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int o = 17 * (4 * g + j);
            v |= ((R[o >> 2] >> (8 * (o & 3))) & 0xFFu) << (8 * j);
        }
        *reinterpret_cast<uint32_t*>(st + offSA + g * 512 + 16 * (r & 31) + 4 * (r >> 5)) = v;
    }
}

// where expert e's weights sit in the weight arrays: its own index, or the
// cache slot that holds it.  The map is read only if the cache header in
// front of it was set up for these sizes (the state buffer is then large
// enough); otherwise, or for a slot outside the arrays, slot 0 is read
// instead and the status word records the error.
__device__ __forceinline__ int weight_slot(const MxArgs& p, int e) {
    if (!p.slot_of) return e;
    const CacheHeader* h = reinterpret_cast<const CacheHeader*>(p.slot_of) - 1;
    if (h->magic != kCacheMagic || h->E != p.E || h->slots != p.nslots) {
        set_error(p.hdr, K3MOE_ERR_INVALID_ARG, 73);
        return 0;
    }
    const int s = p.slot_of[e];
    if (s < 0 || s >= p.nslots) {
        set_error(p.hdr, K3MOE_ERR_INVALID_ARG, 72);
        return 0;
    }
    return s;
}

// The canonical scale rows of a stage (the TMA box puts row r's 16 E8M0 bytes,
// blocks 16 ks .. 16 ks + 15, at byte 16 r) -> the two 512-byte atoms of chunk
// mt (blocks 8 mt .. 8 mt + 3 and 8 mt + 4 .. 8 mt + 7 of the stage), byte
// 16 (m % 32) + 4 (m / 32) + b for row m.  One warp: lane l moves rows l,
// l + 32, l + 64 and l + 96.
__device__ __forceinline__ void relay_sf(const uint8_t* raw, uint8_t* atoms, int mt, int lane) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint2 v = *reinterpret_cast<const uint2*>(raw + 16 * (lane + 32 * q) + 8 * mt);
        *reinterpret_cast<uint32_t*>(atoms + 16 * lane + 4 * q) = v.x;
        *reinterpret_cast<uint32_t*>(atoms + 512 + 16 * lane + 4 * q) = v.y;
    }
}

template <int TERMS, int WF>
__global__ void __launch_bounds__(WF == kWfGgml ? kMxThreads + kGgThreads : kMxThreads, 1)
mx_stream_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA3,
                 const __grid_constant__ CUtensorMap tmS, const __grid_constant__ CUtensorMap tmS3,
                 MxArgs p) {
    constexpr bool GG = WF == kWfGgml;
    constexpr bool CANON = WF == kWfCanon;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    __shared__ __align__(8) uint64_t full[kMaxStages], empty[kMaxStages], acc_full[2], acc_empty[2];
    __shared__ __align__(8) uint64_t raw[GG ? kMaxStages : 1];  // ggml: the stage's copies landed
    __shared__ uint32_t tmem_holder;
    __shared__ int abort_s;
    volatile int* abort_flag = &abort_s;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t NB = static_cast<uint32_t>(p.N) * 128;  // B bytes per chunk
    const uint64_t lim = p.inject ? 1000000ull : kWaitLimitNs;
    const bool drop_first = p.inject && blockIdx.x == 0;
    // stage layout: A chunks | B chunks | SFA atoms (2 per chunk) | SFB atoms
    // [| canonical scale rows]; ggml weights: A chunks | SFA atoms | B chunks |
    // SFB atoms, so that the stage's 17-byte blocks land on the A and SFA bytes
    // they become
    const uint32_t offB = GG ? kStageA + kChunks * 1024 : kStageA;
    const uint32_t offSA = GG ? kStageA : kStageA + kChunks * NB;
    const uint32_t offSB = GG ? offB + kChunks * NB : offSA + kChunks * 1024;
    const uint32_t offRaw = offSB + kChunks * 1024;

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.RS; ++s) {
            mbar_init(&full[s], 1);   // the copies (or, ggml, the converting threads)
            mbar_init(&empty[s], 2);  // one commit per MMA issuer
            if (GG) mbar_init(&raw[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&acc_full[a], 2);
            mbar_init(&acc_empty[a], 4);
        }
        abort_s = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        fence_proxy_async();
    }
    if (warp == 1) tmem_alloc(&tmem_holder, kTmemCols);
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmA);
        if (p.nmat > 1) prefetch_tmap(&tmA3);
        if (CANON) {
            prefetch_tmap(&tmS);
            if (p.nmat > 1) prefetch_tmap(&tmS3);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_holder;

    // The weight loads of the first stages need only the active list.  The down
    // projection may issue them before waiting for the finish kernel: the list
    // was written by the top-k kernel, which completed before the up projection
    // (this grid's predecessor's predecessor) passed its own wait.
    int U = 0, w0 = 0, w1 = 0;
    auto split = [&]() {
        U = *p.count;
        const long long W = static_cast<long long>(U) * p.nmat * p.tiles * p.KS;
        w0 = static_cast<int>(W * blockIdx.x / gridDim.x);
        w1 = static_cast<int>(W * (blockIdx.x + 1) / gridDim.x);
    };
    // stage j of this CTA's range: weight codes and their scales (A side) or the
    // activation codes and scales (B side) into ring slot j % RS
    auto issue_a = [&](const Cursor& c, int e, uint8_t* st, uint64_t* bar) {
        const int c0 = c.ks * kChunks;
        const int nch = min(kChunks, p.KC - c0);
        const CUtensorMap* tm = c.mat == 0 ? &tmA : &tmA3;
        const int y = e * p.rows + c.tile * 128;
        // weights pass through L2 once (the last unit of an expert reads them
        // for the last time), so they are let go first; with several units
        // per expert the earlier reads ask L2 to keep them
        const uint64_t pol = c.grp + 1 < c.ngrp ? l2_policy_evict_last() : l2_policy_evict_first();
        if constexpr (GG) {  // one box of 32-bit words: 128 rows x 272 bytes (K is a multiple of 512)
            tma_load_2d_hint(st, tm, bar, c.ks * (kGgRowBytes / 4), y, pol);
        } else {
            for (int cc = 0; cc < nch; ++cc)
                tma_load_2d_hint(st + cc * kChunkA, tm, bar, (c0 + cc) * 128, y, pol);
            if constexpr (CANON) {  // 16 scale bytes of each of the 128 rows (K is a multiple of 512)
                tma_load_2d_hint(st + offRaw, c.mat == 0 ? &tmS : &tmS3, bar, c.ks * 16, y, pol);
            } else {  // the stage's prepared atoms, consecutive within the tile
                const int g0 = 2 * c0, ng = min(2 * kChunks, p.G - g0);
                bulk_load_hint(st + offSA,
                               p.sf[c.mat] + (static_cast<size_t>(e * p.tiles + c.tile) * p.G + g0) * 512,
                               ng * 512, bar, pol);
            }
        }
    };
    // the activation side of a unit is read again for every row tile of both
    // matrices (48 times at the K3 widths), spread over the unit's whole
    // stream: L2 is asked to keep it while the weights stream past
    auto issue_b = [&](const Cursor& c, uint8_t* st, uint64_t* bar) {
        const int c0 = c.ks * kChunks;
        const int nch = min(kChunks, p.KC - c0);
        const uint64_t pol = l2_policy_evict_last();
        bulk_load_hint(st + offB, p.bq + c.u * p.bq_ustride + static_cast<size_t>(c0) * NB, nch * NB, bar, pol);
        bulk_load_hint(st + offSB, p.bsf + c.u * p.bsf_ustride + static_cast<size_t>(2 * c0) * 512, nch * 1024, bar,
                       pol);
    };
    auto a_bytes = [&](const Cursor& c) {
        if (GG) return static_cast<uint32_t>(kGgStageBytes);
        const int c0 = c.ks * kChunks;
        const int nch = min(kChunks, p.KC - c0);
        const int sfb = CANON ? kRawSf : min(2 * kChunks, p.G - 2 * c0) * 512;
        return static_cast<uint32_t>(nch * kChunkA + sfb);
    };
    // the barrier the stage's copies complete on
    auto ld_bar = [&](int s) { return GG ? &raw[s] : &full[s]; };
    auto b_bytes = [&](const Cursor& c) {
        return static_cast<uint32_t>(min(kChunks, p.KC - c.ks * kChunks)) * (NB + 1024);
    };
    int early = 0;  // stages whose A side was issued before the wait
    if (p.early_a) {
        split();
        if (warp == 0 && lane == 0 && w0 < w1) {
            Cursor c(w0, p);
            early = min(p.RS, w1 - w0);
            for (int j = 0; j < early; ++j) {
                uint8_t* st = smem + static_cast<size_t>(j) * p.stage_bytes;
                mbar_expect_tx_only(ld_bar(j), a_bytes(c));
                issue_a(c, weight_slot(p, p.active[c.u]), st, ld_bar(j));
                c.next(p);
            }
        }
    }
    // the kernel before this one wrote the active list (up) or B (down).  The
    // down pass lets the combine launch at once (it reads nothing before its own
    // wait); the up pass triggers only after its wait, because the down pass
    // reads the active list before waiting and may launch as soon as the finish
    // kernel has started
    if (p.early_a) pdl_trigger();
    pdl_wait();
    if (!p.early_a) pdl_trigger();
    if (!p.early_a) split();
    stamp_start(p.st);

    if (warp == 0) {
        if (lane == 0 && w0 < w1) {
            // ------------------------------ producer ------------------------------
            Cursor c(w0, p);
            int e = weight_slot(p, p.active[c.u]);
            int s = 0;
            uint32_t ph = 0;
            int issued = 0;
            for (int w = w0; w < w1; ++w) {
                uint8_t* st = smem + static_cast<size_t>(s) * p.stage_bytes;
                if (issued < early) {
                    mbar_expect_tx(ld_bar(s), b_bytes(c));  // the arrival of the stage
                    issue_b(c, st, ld_bar(s));
                } else if (drop_first && w == w0) {
                    // test aid: this stage is never signalled, so its consumer's
                    // bounded wait runs out
                } else {
                    if (!mbar_wait(&empty[s], ph ^ 1, abort_flag, p.hdr, 70, lim)) break;
                    mbar_expect_tx(ld_bar(s), a_bytes(c) + b_bytes(c));
                    issue_a(c, e, st, ld_bar(s));
                    issue_b(c, st, ld_bar(s));
                }
                ++issued;
                if (++s == p.RS) {
                    s = 0;
                    ph ^= 1;
                }
                const int u_prev = c.u;
                c.next(p);
                if (c.u != u_prev && w + 1 < w1) e = weight_slot(p, p.active[c.u]);
            }
            // copies still in flight (after an abort) finish before the CTA exits
            for (int j = issued > p.RS ? issued - p.RS : 0; j < issued; ++j) {
                if (drop_first && j == 0) continue;  // nothing was issued for it
                const uint64_t t0 = global_ns();
                while (!mbar_try_wait(ld_bar(j % p.RS), (j / p.RS) & 1) &&
                       global_ns() - t0 < kWaitLimitNs) {
                }
            }
        }
    } else if (warp == 1 || warp == 6) {
        if (w0 < w1) {
            // ------------------------------ MMA issuers ---------------------------
            // lane 0 waits and issues; with canonical scales the whole warp first
            // re-lays its chunk's scale rows into atoms
            const int mt = warp == 1 ? 0 : 1;  // the stage's chunk this warp multiplies
            int ks = Cursor(w0, p).ks;
            int s = 0, seg = 0, ps = 0;
            uint32_t ph = 0, pph = 0;
            const uint32_t id0 = idesc_f4(128, p.N, 0, 0);
            const uint32_t slots = tmem + kSfBase + 128 * mt;
            for (int i = 0, w = w0; w < w1; ++i, ++w) {
                const bool seg_start = (w == w0) || ks == 0;
                const bool seg_end = (w + 1 == w1) || ks == p.KS - 1;
                const int a = seg & 1;
                bool ok = true;
                if (lane == 0) {
                    ok = !seg_start || mbar_wait(&acc_empty[a], ((seg >> 1) & 1) ^ 1, abort_flag, p.hdr, 71, lim);
                    ok = ok && mbar_wait(&full[s], ph, abort_flag, p.hdr, 72, lim);
                    // the scale slots are reused: the previous stage's MMAs have finished
                    ok = ok && (i == 0 || mbar_wait(&empty[ps], pph, abort_flag, p.hdr, 73, lim));
                }
                if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
                if (i > 0 && ++ps == p.RS) {
                    ps = 0;
                    pph ^= 1;
                }
                tc_fence_after();
                const int kv = p.K - (ks * kChunks + mt) * 256;  // inputs of this chunk (<= 0: none)
                if (kv > 0) {
                    uint8_t* stage = smem + static_cast<size_t>(s) * p.stage_bytes;
                    if constexpr (CANON) {
                        relay_sf(stage + offRaw, stage + offSA + 1024 * mt, mt, lane);
                        fence_proxy_async();  // tcgen05.cp reads the atoms through the async proxy
                        __syncwarp();
                    }
                    if (lane == 0) {
                        const uint32_t st = smem_u32(stage);
                        for (int h = 0; h < 2; ++h) {  // the chunk's 128-wide scale groups
                            if (128 * h >= kv) break;
                            tmem_cp_sf(slots + 64 * h, st + offSA + 512 * (2 * mt + h));
                            tmem_cp_sf(slots + 64 * h + 32, st + offSB + 512 * (2 * mt + h));
                        }
                        const uint32_t d_t = tmem + (2 * a + mt) * kMaxN;
                        const uint64_t ad = sw128_desc(st + mt * kChunkA), bd = sw128_desc(st + offB + mt * NB);
                        const int nmma = min(4, kv / 64);
                        for (int j = 0; j < nmma; ++j) {  // K = 64 each: group j / 2, scale id 2 (j % 2)
                            const uint32_t sfa = slots + 64 * (j >> 1);
                            const uint32_t id = static_cast<uint32_t>(2 * (j & 1));
                            mma_f4(d_t, ad + 2 * j, bd + 2 * j, id0 | (id << 4) | (id << 29), sfa, sfa + 32,
                                   (seg_start && j == 0) ? 0u : 1u);
                        }
                    }
                }
                if (lane == 0) {
                    mma_commit(&empty[s]);
                    if (seg_end) mma_commit(&acc_full[a]);
                }
                if (seg_end) ++seg;
                if (++s == p.RS) {
                    s = 0;
                    ph ^= 1;
                }
                if (++ks == p.KS) ks = 0;
            }
        }
    } else if (GG && warp >= kMxThreads / 32) {
        // ------------------------ ggml block conversion -----------------------
        // thread r converts tile row r of every stage, in stage order, and the
        // last of the 128 to finish hands the stage to the MMA issuers
        const int r = threadIdx.x - kMxThreads;
        int s = 0;
        uint32_t ph = 0;
        for (int w = w0; w < w1; ++w) {
            const bool ok = mbar_wait(&raw[s], ph, abort_flag, p.hdr, 76, lim);
            if (!named_bar_and(kGgBar, kGgThreads, ok)) break;
            gg_convert_row(smem + static_cast<size_t>(s) * p.stage_bytes, r, offSA);
            fence_proxy_async();  // the MMA and tcgen05.cp read these bytes through the async proxy
            named_bar_sync(kGgBar, kGgThreads);
            if (r == 0) mbar_arrive(&full[s]);
            if (++s == p.RS) {
                s = 0;
                ph ^= 1;
            }
        }
    } else {
        // ------------------------------ epilogue ---------------------------------
        const int q = warp & 3;  // TMEM lanes 32q .. 32q + 31
        Cursor c(w0 < w1 ? w0 : 0, p);
        int seg = 0;
        for (int w = w0; w < w1;) {
            const int ks_begin = c.ks;
            const int len = min(p.KS - c.ks, w1 - w);
            const bool whole = ks_begin == 0 && len == p.KS;
            const int a = seg & 1;
            if (!__all_sync(0xffffffffu, mbar_wait(&acc_full[a], (seg >> 1) & 1, abort_flag, p.hdr, 74, lim)))
                break;
            tc_fence_after();
            // the second issuer's accumulator holds data unless the segment is only
            // a last stage with a single chunk
            const bool has_d1 = (p.KC % kChunks) == 0 || ks_begin < p.KS - 1;
            float v[kMaxN];
            const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + 2 * a * kMaxN;
#pragma unroll
            for (int c16 = 0; c16 < kMaxN / 16; ++c16) {
                if (c16 * 16 < p.N) {
                    float v16[16];
                    tmem_ld16(taddr + c16 * 16, v16);
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[c16 * 16 + i] = v16[i];
                    if (has_d1) {
                        tmem_ld16(taddr + kMaxN + c16 * 16, v16);
#pragma unroll
                        for (int i = 0; i < 16; ++i) v[c16 * 16 + i] += v16[i];
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[c16 * 16 + i] = 0.0f;
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[a]);
            const int mat = c.mat, mats = p.nmat;
            const int row = c.tile * 128 + q * 32 + lane;
            // rows of the last tile past the expert's own rows belong to the next
            // expert (or lie past the array): computed, never stored
            if (row < p.rows) {
                const size_t plane = static_cast<size_t>(p.umax) * p.T * p.rows_out;
                float* dst = p.part + static_cast<size_t>((ks_begin == 0 ? 0 : 1) * mats + mat) * plane +
                             static_cast<size_t>(c.u) * p.T * p.rows_out + row;
                const int tokens = p.ucnt ? p.ucnt[c.u] : p.T;
#pragma unroll
                for (int t = 0; t < kMaxN / TERMS; ++t) {
                    if (t >= tokens) break;
                    float sum = 0.0f;
#pragma unroll
                    for (int j = 0; j < TERMS; ++j) sum += v[TERMS * t + j];
                    dst[static_cast<size_t>(t) * p.rows_out] = sum;
                    if (whole) dst[static_cast<size_t>(mats) * plane + static_cast<size_t>(t) * p.rows_out] = 0.0f;
                }
            }
            w += len;
            ++seg;
            c.next_segment(p);
        }
    }

    tc_fence_before();
    __syncthreads();
    stamp_end(p.st);
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// One item of the finish step: h = silu(g) * u for 256 hidden columns (chunk
// c) of token t of unit u, from the four partial planes (g slot 0, u slot 0,
// g slot 1, u slot 1, added in that order), quantised to TERMS E2M1 terms in
// the B layout of the down projection.  One warp: lane 4 kb + r takes
// elements 8 r .. 8 r + 7 of 32-block kb; blocks past f (a last partial
// chunk) are never read by the down projection and are not written.
template <int TERMS>
__device__ __forceinline__ void finish_item(const float* __restrict__ part, size_t plane, int T, int f, int N, int u,
                                            int t, int c, uint8_t* __restrict__ hq, uint8_t* __restrict__ hsf,
                                            int lane) {
    const int kb = lane >> 2, r = lane & 3;
    const int KC = (f + 255) / 256;
    const bool in = 256 * c + 32 * kb < f;  // this lane's block exists
    float v[8];
    if (in) {
        const float* g0 = part + (static_cast<size_t>(u) * T + t) * f + 256 * c + 32 * kb + 8 * r;
        float a[8], b[8], cc[8], dd[8];
        *reinterpret_cast<float4*>(a) = *reinterpret_cast<const float4*>(g0);
        *reinterpret_cast<float4*>(a + 4) = *reinterpret_cast<const float4*>(g0 + 4);
        *reinterpret_cast<float4*>(b) = *reinterpret_cast<const float4*>(g0 + plane);
        *reinterpret_cast<float4*>(b + 4) = *reinterpret_cast<const float4*>(g0 + plane + 4);
        *reinterpret_cast<float4*>(cc) = *reinterpret_cast<const float4*>(g0 + 2 * plane);
        *reinterpret_cast<float4*>(cc + 4) = *reinterpret_cast<const float4*>(g0 + 2 * plane + 4);
        *reinterpret_cast<float4*>(dd) = *reinterpret_cast<const float4*>(g0 + 3 * plane);
        *reinterpret_cast<float4*>(dd + 4) = *reinterpret_cast<const float4*>(g0 + 3 * plane + 4);
#pragma unroll
        for (int q = 0; q < 8; ++q) v[q] = silu_f32(a[q] + cc[q]) * (b[q] + dd[q]);
    } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) v[q] = 0.0f;
    }
    uint32_t w[TERMS], sb[TERMS];
    quantize8_terms<TERMS>(v, w, sb);  // shuffles stay within the block's four lanes
    if (!in) return;
    uint8_t* codes = hq + (static_cast<size_t>(u) * KC + c) * N * 128;
    uint8_t* scales = hsf + (static_cast<size_t>(u) * KC + c) * 1024;
#pragma unroll
    for (int j = 0; j < TERMS; ++j) {
        const int n = TERMS * t + j;
        *reinterpret_cast<uint32_t*>(codes + n * 128 + ((kb ^ (n & 7)) << 4) + 4 * r) = w[j];
        if (r == 0) scales[(kb >> 2) * 512 + sf_atom_offset(n, kb & 3)] = static_cast<uint8_t>(sb[j]);
    }
}

// The finish step: one warp per (unit, token, 256-wide chunk), grid-strided
// over the units (the grid is sized for the SMs, not for the largest possible
// number of units).  Tokens a unit does not have are skipped: their MMA
// columns are never read.
template <int TERMS>
__global__ void __launch_bounds__(256)
mx_finish_kernel(const float* __restrict__ part, int umax, int T, int f, int N,
                 const int32_t* __restrict__ count, const int32_t* __restrict__ ucnt, uint8_t* __restrict__ hq,
                 uint8_t* __restrict__ hsf, uint64_t* st) {
    // the down projection may launch now: its CTAs start on the SMs the up
    // projection frees and issue their first weight loads during this kernel
    // (this grid was launched after every up CTA passed its wait, so the active
    // list they read is final)
    pdl_trigger();
    pdl_wait();
    StampScope stamp(st);
    const int lane = threadIdx.x & 31;
    const int KC = (f + 255) / 256;
    const int items = *count * T * KC;
    const size_t plane = static_cast<size_t>(umax) * T * f;
    for (int i = blockIdx.x * 8 + (threadIdx.x >> 5); i < items; i += gridDim.x * 8) {
        const int u = i / (T * KC);
        const int rr = i - u * T * KC;
        const int t = rr / KC, c = rr - t * KC;
        if (ucnt && t >= ucnt[u]) continue;
        finish_item<TERMS>(part, plane, T, f, N, u, t, c, hq, hsf, lane);
    }
}

// Token rows (bf16) -> kTerms E2M1 terms in the B layout (used when the
// router did not write them).  One warp per (token, 32-block).
__global__ void __launch_bounds__(256)
mx_quantize_rows_kernel(const uint16_t* __restrict__ x, int T, int K, int N, uint8_t* __restrict__ xq,
                        uint8_t* __restrict__ xsf, uint64_t* st) {
    pdl_wait();
    pdl_trigger();
    StampScope stamp(st);
    const int lane = threadIdx.x & 31;
    const int nb = K / 32;
    const int i = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (i >= T * nb) return;
    const int t = i / nb, b = i - t * nb;
    uint32_t q[kTerms], sb[kTerms];
    quantize_terms(bf16_to_f32(x[static_cast<size_t>(t) * K + 32 * b + lane]), q, sb);
    store_terms(q, sb, t, b & 7, xq + static_cast<size_t>(b >> 3) * N * 128,
                xsf + static_cast<size_t>(b >> 3) * 1024);
}

// out[t, :] = bf16(sum_j w[t, j] * (y0 + y1)[unit(idx[t, j]), t, :]), j in slot
// order; the unit of an expert is its position in the active list.  A CTA
// owns 128 columns of one token: its 8 warps load the k slots' rows at once
// (warp g takes slots g, g + 8, ...; a lane takes 4 columns), park the
// weighted rows in shared memory, and one thread per column adds them in
// slot order.
constexpr int kCombineThreads = 256;
constexpr int kCombineCols = 128;
constexpr int kCombineMaxUnits = 256;  // decode: T * k <= 8 * 32

__global__ void __launch_bounds__(kCombineThreads)
mx_combine_kernel(const float* __restrict__ y, int umax, int T, int d, const float* __restrict__ wts,
                  const int32_t* __restrict__ idx, const int32_t* __restrict__ active, int E, int k,
                  const int32_t* __restrict__ rowmap, uint16_t* __restrict__ out, uint64_t* st) {
    __shared__ int rows[32];
    __shared__ float wk[32];
    __shared__ int act[kCombineMaxUnits];
    __shared__ __align__(16) float part[32][kCombineCols];
    // The selection, its weights and the unit lists were final before this
    // grid could launch: it launches only after the down pass has started,
    // the down pass only after the finish kernel has started, and the finish
    // kernel only after the up pass has passed its own wait, which returns
    // once the top-k (or unit listing) kernel has completed.  The rows are
    // looked up before the wait for the down pass.
    const int t = blockIdx.y;
    const int lane = threadIdx.x & 31, g = threadIdx.x >> 5;
    if (rowmap) {
        // unit-grouped: the row of every (token, slot) pair was listed with the units
        if (threadIdx.x < k) {
            rows[threadIdx.x] = rowmap[t * k + threadIdx.x];
            wk[threadIdx.x] = wts[t * k + threadIdx.x];
        }
    } else {
        const int U = active[E];
        for (int i = threadIdx.x; i < U; i += blockDim.x) act[i] = active[i];
        __syncthreads();
        if (threadIdx.x < k) {
            const int e = idx[t * k + threadIdx.x];
            int lo = 0, hi = U - 1;
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (act[mid] < e) lo = mid + 1;
                else hi = mid;
            }
            rows[threadIdx.x] = lo * T + t;
            wk[threadIdx.x] = wts[t * k + threadIdx.x];
        }
    }
    __syncthreads();
    pdl_wait();  // y is the down pass's output
    pdl_trigger();
    StampScope stamp(st);
    const int c0 = blockIdx.x * kCombineCols;
    const size_t slot = static_cast<size_t>(umax) * T * d;
    if (c0 + lane * 4 < d) {
#pragma unroll 4
        for (int j = g; j < k; j += kCombineThreads / 32) {
            const float* yr = y + static_cast<size_t>(rows[j]) * d + c0 + lane * 4;
            const float4 v = *reinterpret_cast<const float4*>(yr);
            const float4 v2 = *reinterpret_cast<const float4*>(yr + slot);
            const float w = wk[j];
            *reinterpret_cast<float4*>(&part[j][lane * 4]) =
                make_float4(w * (v.x + v2.x), w * (v.y + v2.y), w * (v.z + v2.z), w * (v.w + v2.w));
        }
    }
    __syncthreads();
    const int c = c0 + threadIdx.x;
    if (threadIdx.x < kCombineCols && c < d) {
        float acc = 0.0f;
        for (int j = 0; j < k; ++j) acc += part[j][threadIdx.x];
        out[static_cast<size_t>(t) * d + c] = f32_to_bf16(acc);
    }
}

// ---------------------------------------------------------------------------
// Unit-grouped streaming (more tokens than the decode path takes, few per
// expert): every expert's sorted token list (from the permutation) is cut into
// units of at most kUnitTokens tokens, and the streaming kernels run over the
// units exactly as the decode path runs over the active experts, with each
// unit's own token rows as the B operand.  An expert's weights are read once
// per unit.
// ---------------------------------------------------------------------------
// Units take four E2M1 terms per token (16 tokens within N = 64; an expert's
// output within about 1.1e-3 of its RMS instead of 1.2e-4 with five), so that
// most experts need a single unit at a few hundred tokens.
constexpr int kUnitTerms = 4;
constexpr int kUnitTokens = kMaxN / kUnitTerms;  // 16

// Unit list and the expert-output row of every (token, slot) pair.  One CTA of
// 1024 threads (E <= 1024): units of expert e are ubase[e] .. ubase[e + 1) - 1.
__global__ void __launch_bounds__(1024)
mx_units_kernel(const int32_t* __restrict__ counts, const int32_t* __restrict__ offsets,
                const int32_t* __restrict__ idx, const int32_t* __restrict__ inv, int E, int P,
                int32_t* __restrict__ unit_exp, int32_t* __restrict__ unit_row0, int32_t* __restrict__ unit_cnt,
                int32_t* __restrict__ nunits, int32_t* __restrict__ rowmap, int32_t* __restrict__ ubase_out,
                uint64_t* st) {
    StampScope stamp(st);
    __shared__ int ubase[1024 + 1];
    __shared__ int warp_tot[32];
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int n = tid < E ? (counts[tid] + kUnitTokens - 1) / kUnitTokens : 0;
    int incl = n;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) warp_tot[wid] = incl;
    __syncthreads();
    if (wid == 0) {
        int w = warp_tot[lane], wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += v;
        }
        warp_tot[lane] = wi - w;  // exclusive over warps
    }
    __syncthreads();
    const int excl = warp_tot[wid] + incl - n;
    if (tid < E) ubase[tid] = excl;
    if (tid == blockDim.x - 1) ubase[E] = excl + n;  // blockDim.x >= E: the last thread sees the total
    __syncthreads();
    const int U = ubase[E];
    if (tid == 0) *nunits = U;
    for (int e = tid; e <= E; e += blockDim.x) ubase_out[e] = ubase[e];
    for (int i = tid; i < U; i += blockDim.x) {
        int lo = 0, hi = E - 1;  // expert of unit i: largest e with ubase[e] <= i
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (ubase[mid] <= i) lo = mid;
            else hi = mid - 1;
        }
        const int g = i - ubase[lo];
        unit_exp[i] = lo;
        unit_row0[i] = offsets[lo] + g * kUnitTokens;
        unit_cnt[i] = min(kUnitTokens, counts[lo] - g * kUnitTokens);
    }
    for (int q = tid; q < P; q += blockDim.x) {
        const int e = idx[q];
        const int local = inv[q] - offsets[e];
        rowmap[q] = (ubase[e] + local / kUnitTokens) * kUnitTokens + local % kUnitTokens;
    }
}

// Token rows as kUnitTerms E2M1 terms, once per token (unswizzled): codes
// [t][term][K / 2] (element 2i in the low nibble), E8M0 scales [t][term][K / 32].
// One warp per (token, 256-wide chunk), lane 4 kb + r taking elements 8 r ..
// 8 r + 7 of 32-block kb (blocks past K, in a last partial chunk, idle);
// grid-strided.
__global__ void __launch_bounds__(256)
mx_token_terms_kernel(const uint16_t* __restrict__ x, int T, int K, uint8_t* __restrict__ tq,
                      uint8_t* __restrict__ tsf, uint64_t* st) {
    StampScope stamp(st);
    const int lane = threadIdx.x & 31, kb = lane >> 2, r = lane & 3;
    const int KC = (K + 255) / 256, nb = K / 32;
    for (int i = blockIdx.x * 8 + (threadIdx.x >> 5); i < T * KC; i += gridDim.x * 8) {
        const int t = i / KC, c = i - t * KC;
        const bool in = 256 * c + 32 * kb < K;
        const uint4 raw = in ? *reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * K + 256 * c + 32 * kb + 8 * r)
                             : make_uint4(0, 0, 0, 0);
        const uint32_t wr[4] = {raw.x, raw.y, raw.z, raw.w};
        float v[8];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            v[2 * q] = __uint_as_float(wr[q] << 16);
            v[2 * q + 1] = __uint_as_float(wr[q] & 0xFFFF0000u);
        }
        uint32_t w[kUnitTerms], sb[kUnitTerms];
        quantize8_terms<kUnitTerms>(v, w, sb);
        if (!in) continue;
#pragma unroll
        for (int j = 0; j < kUnitTerms; ++j) {
            const size_t row = static_cast<size_t>(t) * kUnitTerms + j;
            *reinterpret_cast<uint32_t*>(tq + row * (K / 2) + 128 * c + 16 * kb + 4 * r) = w[j];
            if (r == 0) tsf[row * nb + 8 * c + kb] = static_cast<uint8_t>(sb[j]);
        }
    }
}

// B operand of the unit-grouped up projection: the term rows of token i of
// unit u (sorted row unit_row0[u] + i) copied into the unit's swizzled layout;
// tokens past unit_cnt[u] are left as they are (their MMA columns are never
// read).  One thread per (unit, token, term, 32-block), grid-strided.
__global__ void __launch_bounds__(256)
mx_unit_terms_kernel(const uint8_t* __restrict__ tq, const uint8_t* __restrict__ tsf,
                     const int32_t* __restrict__ perm, int k, int K, int N, const int32_t* __restrict__ nunits,
                     const int32_t* __restrict__ unit_row0, const int32_t* __restrict__ unit_cnt,
                     uint8_t* __restrict__ bq, uint8_t* __restrict__ bsf, uint64_t* st) {
    StampScope stamp(st);
    const int nb = K / 32, KC = (K + 255) / 256;
    const int per_unit = kUnitTokens * kUnitTerms * nb;
    const long long items = static_cast<long long>(*nunits) * per_unit;
    for (long long it = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; it < items;
         it += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int u = static_cast<int>(it / per_unit);
        int r = static_cast<int>(it - static_cast<long long>(u) * per_unit);
        const int i = r / (kUnitTerms * nb);
        r -= i * kUnitTerms * nb;
        const int j = r / nb, b = r - j * nb;
        if (i >= unit_cnt[u]) continue;
        const int tok = perm[unit_row0[u] + i] / k;
        const size_t src = static_cast<size_t>(tok) * kUnitTerms + j;
        const int n = kUnitTerms * i + j, c = b >> 3, g = b & 7;
        const size_t cb = static_cast<size_t>(u) * KC + c;
        *reinterpret_cast<uint4*>(bq + cb * N * 128 + n * 128 + ((g ^ (n & 7)) << 4)) =
            *reinterpret_cast<const uint4*>(tq + src * (K / 2) + 16 * b);
        bsf[cb * 1024 + (g >> 2) * 512 + sf_atom_offset(n, g & 3)] = tsf[src * nb + b];
    }
}

// ---------------------------------------------------------------------------
// Prepared scale-factor layout.  For a weight matrix of E experts with R rows
// each (a multiple of 64) and K inputs (a multiple of 64), every expert's E8M0
// bytes are grouped per tile of 128 rows (ceil(R / 128) tiles, the last padded
// with zero rows) and 128-wide input group (ceil(K / 128) groups, the last
// padded with zero blocks) into 512-byte atoms: byte 16 (m % 32) + 4 (m / 32)
// + b holds row m of the tile and block b of the group.  The atom of (expert,
// tile, group) starts at ((e * tiles + tile) * groups + group) * 512.  One
// thread per 4-byte word of the atoms (the four blocks of one row and group);
// the padding is written as zeros and skipped by the inverse.
// ---------------------------------------------------------------------------
__global__ void prepare_sf_kernel(uint8_t* __restrict__ canon, int64_t n_words, int R, int K,
                                  uint8_t* __restrict__ atoms, int inverse, uint64_t* st) {
    StampScope stamp(st);
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= n_words) return;
    const int G = (K + 127) / 128, tiles = (R + 127) / 128, nb = K / 32;
    const int64_t atom = i / 128;            // 128 words per atom
    const int wi = static_cast<int>(i - atom * 128);
    const int g = static_cast<int>(atom % G);
    const int64_t et = atom / G;             // e * tiles + tile
    const int64_t e = et / tiles;
    const int tile = static_cast<int>(et - e * tiles);
    const int r = wi >> 2, qd = wi & 3;      // word at byte 16 r + 4 qd: row m = 32 qd + r
    const int row = tile * 128 + 32 * qd + r;
    uint8_t* aw = atoms + atom * 512 + 16 * r + 4 * qd;
    uint8_t* cw = canon + (e * R + row) * nb + 4 * g;
    const int nbv = row < R ? min(4, nb - 4 * g) : 0;  // blocks of this word inside the matrix
    if (inverse) {
        for (int b = 0; b < nbv; ++b) cw[b] = aw[b];
    } else {
        uint32_t w = 0;
        for (int b = 0; b < nbv; ++b) w |= static_cast<uint32_t>(cw[b]) << (8 * b);
        *reinterpret_cast<uint32_t*>(aw) = w;
    }
}

}  // namespace

size_t prepared_sf_bytes(int64_t E, int R, int K) {
    return static_cast<size_t>(E) * ((R + 127) / 128) * ((K + 127) / 128) * 512;
}

cudaError_t launch_prepare_sf(const uint8_t* canon, int64_t E, int R, int K, uint8_t* atoms, int inverse,
                              cudaStream_t s) {
    const int64_t n_words = static_cast<int64_t>(prepared_sf_bytes(E, R, K) / 4);
    if (n_words <= 0) return cudaSuccess;
    const int64_t blocks = (n_words + 255) / 256;
    prepare_sf_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(
        const_cast<uint8_t*>(canon), n_words, R, K, atoms, inverse, trace_stamp(inverse ? "unprepare_sf" : "prepare_sf"));
    trace_mark(inverse ? "unprepare_sf" : "prepare_sf", s);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// host: decode forward
// ---------------------------------------------------------------------------
namespace {

int mx_n(int T, int terms = kTerms) { return (terms * T + 15) / 16 * 16; }
int kc256(int K) { return (K + 255) / 256; }

struct MxScratch {
    uint8_t *xq, *xsf, *hq, *hsf;
    float *up, *y;
    int umax, N;
    size_t bytes;
};

// the B operand takes one 256-wide chunk per 256 inputs (the last may be
// partial): N rows x 128 bytes of codes and 1024 bytes of scale atoms each
MxScratch mx_carve(void* scratch, int T, int E, int k, int d, int f) {
    MxScratch m{};
    m.umax = std::min(E, T * k);
    m.N = mx_n(T);
    char* b = static_cast<char*>(scratch);
    size_t o = 0;
    auto take = [&](size_t bytes) {
        char* r = b ? b + o : nullptr;
        o += align_up(bytes);
        return r;
    };
    const size_t U = static_cast<size_t>(m.umax);
    m.xq = reinterpret_cast<uint8_t*>(take(static_cast<size_t>(kc256(d)) * m.N * 128));
    m.xsf = reinterpret_cast<uint8_t*>(take(static_cast<size_t>(kc256(d)) * 1024));
    m.up = reinterpret_cast<float*>(take(4 * U * T * f * 4));
    m.hq = reinterpret_cast<uint8_t*>(take(U * kc256(f) * m.N * 128));
    m.hsf = reinterpret_cast<uint8_t*>(take(U * kc256(f) * 1024));
    m.y = reinterpret_cast<float*>(take(2 * U * T * d * 4));
    m.bytes = o;
    return m;
}

// stage size and ring depth of the streaming kernels for a B operand of N rows
void ring_shape(MxArgs* p, int wf) {
    const size_t raw = wf == kWfCanon ? kRawSf : 0;
    p->stage_bytes = static_cast<uint32_t>(align_up(kStageA + kChunks * (p->N * 128 + 2048) + raw, 1024));
    p->RS = std::min(kMaxStages, static_cast<int>((226 * 1024) / p->stage_bytes));
}

template <int TERMS, int WF>
cudaError_t launch_stream(const CUtensorMap& a, const CUtensorMap& a3, const CUtensorMap& sc,
                          const CUtensorMap& sc3, MxArgs p, int grid, cudaStream_t s, const char* name) {
    ring_shape(&p, WF);
    if (p.RS < 2 || p.N > kMaxN) return cudaErrorNotSupported;
    const size_t smem = 1024 + static_cast<size_t>(p.RS) * p.stage_bytes;
    // the attribute is per device: raise it once per device to the largest
    // ring any call asks for (not inside graph captures in practice: the
    // first forward runs uncaptured)
    static std::atomic<int> set_bytes[64];
    int dev = 0;
    cudaGetDevice(&dev);
    std::atomic<int>& cur = set_bytes[dev & 63];
    if (cur.load() < static_cast<int>(smem)) {
        const cudaError_t e = cudaFuncSetAttribute(mx_stream_kernel<TERMS, WF>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        cur.store(static_cast<int>(smem));
    }
    p.st = trace_stamp(name);
    const cudaError_t e = launch_pdl(mx_stream_kernel<TERMS, WF>, dim3(grid),
                                     dim3(WF == kWfGgml ? kMxThreads + kGgThreads : kMxThreads), smem, s, a, a3,
                                     sc, sc3, p);
    trace_mark(name, s);
    return e;
}

// Tensor maps of the three matrices over `nslots` expert slots.  Compressed-
// tensors codes: [slots * rows, K / 2] bytes, boxes of 128 bytes (256 inputs)
// x 128 rows, 128-byte swizzle (a box past the end of a row, K % 256 != 0, or
// past the last row is zero-filled).  Canonical E8M0 rows: [slots * rows,
// K / 32] bytes, boxes of 16 bytes (one 512-input stage) x 128 rows, no
// swizzle (rows must be whole 16-byte units: K % 512 == 0).  ggml blocks:
// [slots * rows, K / 32 * 17] bytes as 32-bit words, boxes of 68 words (one
// 512-input stage) x 128 rows, no swizzle (the converting threads swizzle).
struct WeightMaps {
    CUtensorMap q[3], sc[3];  // W1, W3, W2
    int wf;
};

bool make_weight_maps(const uint8_t* const w_q[3], const uint8_t* const w_s[3], int sf_canon, int ggml, int d,
                      int f, uint64_t nslots, WeightMaps* m) {
    m->wf = ggml ? kWfGgml : (sf_canon ? kWfCanon : kWfAtoms);
    for (int i = 0; i < 3; ++i) {
        const uint64_t K = i < 2 ? d : f, rows = nslots * (i < 2 ? f : d);
        bool ok;
        if (ggml) {
            const uint64_t rb = K / 32 * 17;
            ok = make_tmap_rows(&m->q[i], w_q[i], CU_TENSOR_MAP_DATA_TYPE_UINT32, rb, rb / 4, rows, kGgRowBytes / 4,
                                128, CU_TENSOR_MAP_SWIZZLE_NONE);
        } else {
            ok = make_tmap_rows(&m->q[i], w_q[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, K / 2, K / 2, rows, 128, 128,
                                CU_TENSOR_MAP_SWIZZLE_128B);
        }
        if (!ok) return false;
        if (m->wf == kWfCanon) {
            if (K % 512) return false;
            if (!make_tmap_rows(&m->sc[i], w_s[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, K / 32, K / 32, rows, 16, 128,
                                CU_TENSOR_MAP_SWIZZLE_NONE))
                return false;
        } else {
            m->sc[i] = m->q[i];  // unused
        }
    }
    return true;
}

template <int TERMS>
cudaError_t launch_stream_wf(const WeightMaps& wm, bool up, const MxArgs& p, int grid, cudaStream_t s,
                             const char* name) {
    const CUtensorMap& a = wm.q[up ? 0 : 2];
    const CUtensorMap& a3 = wm.q[up ? 1 : 2];
    const CUtensorMap& sc = wm.sc[up ? 0 : 2];
    const CUtensorMap& sc3 = wm.sc[up ? 1 : 2];
    switch (wm.wf) {
        case kWfGgml: return launch_stream<TERMS, kWfGgml>(a, a3, sc, sc3, p, grid, s, name);
        case kWfCanon: return launch_stream<TERMS, kWfCanon>(a, a3, sc, sc3, p, grid, s, name);
        default: return launch_stream<TERMS, kWfAtoms>(a, a3, sc, sc3, p, grid, s, name);
    }
}

// The fields of an up (W1, W3) and a down (W2) pass over units that share B
// layouts of N rows: everything but the unit lists, B pointers and outputs.
void pass_shapes(MxArgs* up, MxArgs* dn, const uint8_t* const w_s[3], int E, int d, int f, int N) {
    up->sf[0] = w_s[0];
    up->sf[1] = w_s[1];
    up->nmat = 2;
    up->E = E;
    up->rows = f;
    up->tiles = (f + 127) / 128;
    up->K = d;
    up->KC = kc256(d);
    up->KS = (up->KC + kChunks - 1) / kChunks;
    up->G = (d + 127) / 128;
    up->N = N;
    up->rows_out = f;
    *dn = *up;
    dn->sf[0] = w_s[2];
    dn->sf[1] = w_s[2];
    dn->nmat = 1;
    dn->early_a = 1;
    dn->rows = d;
    dn->tiles = (d + 127) / 128;
    dn->K = f;
    dn->KC = kc256(f);
    dn->KS = (dn->KC + kChunks - 1) / kChunks;
    dn->G = (f + 127) / 128;
    dn->rows_out = d;
}

}  // namespace

size_t mx_decode_scratch_bytes(int T, int E, int k, int d, int f) {
    return mx_carve(nullptr, T, E, k, d, f).bytes;
}

void mx_decode_xq_slots(void* scratch, int T, int E, int k, int d, int f, uint8_t** xq, uint8_t** xsf,
                        int* N) {
    const MxScratch m = mx_carve(scratch, T, E, k, d, f);
    *xq = m.xq;
    *xsf = m.xsf;
    *N = m.N;
}


cudaError_t launch_mx_decode(const MxDecodeArgs& a, cudaStream_t s) {
    const MxScratch m = mx_carve(a.scratch, a.T, a.E, a.k, a.d, a.f);
    cudaError_t e;
    if (!a.xq_ready) {
        const int warps = a.T * (a.d / 32);
        e = launch_pdl(mx_quantize_rows_kernel, dim3((warps + 7) / 8), dim3(256), 0, s, a.x, a.T, a.d, m.N,
                       m.xq, m.xsf, trace_stamp("quantize_x"));
        trace_mark("quantize_x", s);
        if (e != cudaSuccess) return e;
    }
    // A operands over a slot per expert, or over the cache's slots
    const uint64_t nslots = a.slot_of ? static_cast<uint64_t>(a.nslots) : static_cast<uint64_t>(a.E);
    const uint8_t* const wq[3] = {a.w1_q, a.w3_q, a.w2_q};
    const uint8_t* const ws[3] = {a.w1_sf, a.w3_sf, a.w2_sf};
    WeightMaps wm;
    if (!make_weight_maps(wq, ws, a.sf_canon, a.ggml, a.d, a.f, nslots, &wm)) return cudaErrorNotSupported;

    MxArgs up{}, dn{};
    pass_shapes(&up, &dn, ws, a.E, a.d, a.f, m.N);
    up.bq = m.xq;
    up.bsf = m.xsf;
    up.active = a.active;
    up.count = a.active + a.E;
    up.slot_of = a.slot_of;
    up.nslots = static_cast<int>(nslots);
    up.T = a.T;
    up.part = m.up;
    up.umax = m.umax;
    up.hdr = a.hdr;
    up.inject = a.inject;
    dn.bq = m.hq;
    dn.bsf = m.hsf;
    dn.bq_ustride = static_cast<size_t>(kc256(a.f)) * m.N * 128;
    dn.bsf_ustride = static_cast<size_t>(kc256(a.f)) * 1024;
    dn.active = up.active;
    dn.count = up.count;
    dn.slot_of = up.slot_of;
    dn.nslots = up.nslots;
    dn.T = up.T;
    dn.part = m.y;
    dn.umax = m.umax;
    dn.hdr = a.hdr;

    // every CTA's range must be at least one tile long: at least k experts are active
    const int grid_up = std::min(a.num_sms, a.k * up.nmat * up.tiles);
    if ((e = launch_stream_wf<kTerms>(wm, true, up, grid_up, s, "decode_up"))) return e;

    const int warps = m.umax * a.T * kc256(a.f);
    const int fgrid = std::min((warps + 7) / 8, 8 * a.num_sms);
    e = launch_pdl(mx_finish_kernel<kTerms>, dim3(fgrid), dim3(256), 0, s, static_cast<const float*>(m.up),
                   m.umax, a.T, a.f, m.N, a.active + a.E, static_cast<const int32_t*>(nullptr), m.hq, m.hsf,
                   trace_stamp("decode_finish_up"));
    trace_mark("decode_finish_up", s);
    if (e != cudaSuccess) return e;

    const int grid_dn = std::min(a.num_sms, a.k * dn.tiles);
    if ((e = launch_stream_wf<kTerms>(wm, false, dn, grid_dn, s, "decode_down"))) return e;

    dim3 cgrid((a.d + kCombineCols - 1) / kCombineCols, a.T);
    e = launch_pdl(mx_combine_kernel, cgrid, dim3(kCombineThreads), 0, s, static_cast<const float*>(m.y),
                   m.umax, a.T, a.d, a.wts, a.idx, a.active, a.E, a.k, static_cast<const int32_t*>(nullptr), a.out,
                   trace_stamp("combine"));
    trace_mark("combine", s);
    return e;
}

// ---------------------------------------------------------------------------
// host: unit-grouped streaming forward
// ---------------------------------------------------------------------------
namespace {

struct MxUnitScratch {
    int32_t *unit_exp, *unit_row0, *unit_cnt, *nunits, *rowmap, *ubase;
    uint8_t *tq, *tsf, *xq, *xsf, *hq, *hsf;
    float *up, *y;
    int umax, N;
    size_t bytes;
};

// units <= min(T k, (T k + E (G - 1)) / G): ceil(c / G) <= (c + G - 1) / G per expert
MxUnitScratch mx_units_carve(void* scratch, int T, int E, int k, int d, int f) {
    MxUnitScratch m{};
    const long long P = static_cast<long long>(T) * k;
    m.umax = static_cast<int>(std::min<long long>(P, (P + static_cast<long long>(E) * (kUnitTokens - 1)) / kUnitTokens));
    m.N = mx_n(kUnitTokens, kUnitTerms);
    char* b = static_cast<char*>(scratch);
    size_t o = 0;
    auto take = [&](size_t bytes) {
        char* r = b ? b + o : nullptr;
        o += align_up(bytes);
        return r;
    };
    const size_t U = static_cast<size_t>(m.umax);
    m.unit_exp = reinterpret_cast<int32_t*>(take(U * 4));
    m.unit_row0 = reinterpret_cast<int32_t*>(take(U * 4));
    m.unit_cnt = reinterpret_cast<int32_t*>(take(U * 4));
    m.nunits = reinterpret_cast<int32_t*>(take(4));
    m.ubase = reinterpret_cast<int32_t*>(take(static_cast<size_t>(E + 1) * 4));
    m.rowmap = reinterpret_cast<int32_t*>(take(static_cast<size_t>(P) * 4));
    m.tq = reinterpret_cast<uint8_t*>(take(static_cast<size_t>(T) * kUnitTerms * (d / 2)));
    m.tsf = reinterpret_cast<uint8_t*>(take(static_cast<size_t>(T) * kUnitTerms * (d / 32)));
    m.xq = reinterpret_cast<uint8_t*>(take(U * kc256(d) * m.N * 128));
    m.xsf = reinterpret_cast<uint8_t*>(take(U * kc256(d) * 1024));
    m.up = reinterpret_cast<float*>(take(4 * U * kUnitTokens * f * 4));
    m.hq = reinterpret_cast<uint8_t*>(take(U * kc256(f) * m.N * 128));
    m.hsf = reinterpret_cast<uint8_t*>(take(U * kc256(f) * 1024));
    m.y = reinterpret_cast<float*>(take(2 * U * kUnitTokens * d * 4));
    m.bytes = o;
    return m;
}

}  // namespace

size_t mx_units_scratch_bytes(int T, int E, int k, int d, int f) {
    return mx_units_carve(nullptr, T, E, k, d, f).bytes;
}

cudaError_t launch_mx_units(const MxUnitsArgs& a, cudaStream_t s) {
    const MxUnitScratch m = mx_units_carve(a.scratch, a.T, a.E, a.k, a.d, a.f);
    if (a.E > 1024) return cudaErrorNotSupported;
    const int P = a.T * a.k;
    mx_units_kernel<<<1, 1024, 0, s>>>(a.counts, a.offsets, a.idx, a.inv, a.E, P, m.unit_exp, m.unit_row0,
                                       m.unit_cnt, m.nunits, m.rowmap, m.ubase, trace_stamp("units"));
    trace_mark("units", s);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const long long twarps = static_cast<long long>(a.T) * kc256(a.d);
    mx_token_terms_kernel<<<static_cast<int>(std::min<long long>((twarps + 7) / 8, 8LL * a.num_sms)), 256, 0, s>>>(
        a.x, a.T, a.d, m.tq, m.tsf, trace_stamp("token_terms"));
    trace_mark("token_terms", s);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const long long citems = static_cast<long long>(m.umax) * kUnitTokens * kUnitTerms * (a.d / 32);
    mx_unit_terms_kernel<<<static_cast<int>(std::min<long long>((citems + 255) / 256, 8LL * a.num_sms)), 256, 0,
                           s>>>(m.tq, m.tsf, a.perm, a.k, a.d, m.N, m.nunits, m.unit_row0, m.unit_cnt, m.xq, m.xsf,
                                trace_stamp("unit_terms"));
    trace_mark("unit_terms", s);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;

    const uint64_t nslots = a.slot_of ? static_cast<uint64_t>(a.nslots) : static_cast<uint64_t>(a.E);
    const uint8_t* const wq[3] = {a.w1_q, a.w3_q, a.w2_q};
    const uint8_t* const ws[3] = {a.w1_sf, a.w3_sf, a.w2_sf};
    WeightMaps wm;
    if (!make_weight_maps(wq, ws, a.sf_canon, a.ggml, a.d, a.f, nslots, &wm)) return cudaErrorNotSupported;

    MxArgs up{}, dn{};
    pass_shapes(&up, &dn, ws, a.E, a.d, a.f, m.N);
    up.bq = m.xq;
    up.bsf = m.xsf;
    up.bq_ustride = static_cast<size_t>(kc256(a.d)) * m.N * 128;
    up.bsf_ustride = static_cast<size_t>(kc256(a.d)) * 1024;
    up.active = m.unit_exp;
    up.count = m.nunits;
    up.ucnt = m.unit_cnt;
    up.ubase = m.ubase;
    up.slot_of = a.slot_of;
    up.nslots = static_cast<int>(nslots);
    up.T = kUnitTokens;
    up.part = m.up;
    up.umax = m.umax;
    up.hdr = a.hdr;
    up.inject = a.inject;
    // every CTA's range must be at least one tile long: there are at least k units
    const int grid_up = std::min(a.num_sms, a.k * up.nmat * up.tiles);
    if ((e = launch_stream_wf<kUnitTerms>(wm, true, up, grid_up, s, "units_up"))) return e;

    const long long fwarps = static_cast<long long>(m.umax) * kUnitTokens * kc256(a.f);
    const int fgrid = static_cast<int>(std::min<long long>((fwarps + 7) / 8, 8LL * a.num_sms));
    e = launch_pdl(mx_finish_kernel<kUnitTerms>, dim3(fgrid), dim3(256), 0, s, static_cast<const float*>(m.up), m.umax,
                   kUnitTokens, a.f, m.N, static_cast<const int32_t*>(m.nunits),
                   static_cast<const int32_t*>(m.unit_cnt), m.hq, m.hsf, trace_stamp("units_finish_up"));
    trace_mark("units_finish_up", s);
    if (e != cudaSuccess) return e;

    dn.bq = m.hq;
    dn.bsf = m.hsf;
    dn.bq_ustride = static_cast<size_t>(kc256(a.f)) * m.N * 128;
    dn.bsf_ustride = static_cast<size_t>(kc256(a.f)) * 1024;
    dn.active = up.active;
    dn.count = up.count;
    dn.ucnt = up.ucnt;
    dn.ubase = up.ubase;
    dn.slot_of = up.slot_of;
    dn.nslots = up.nslots;
    dn.T = up.T;
    dn.part = m.y;
    dn.umax = m.umax;
    dn.hdr = a.hdr;
    const int grid_dn = std::min(a.num_sms, a.k * dn.tiles);
    if ((e = launch_stream_wf<kUnitTerms>(wm, false, dn, grid_dn, s, "units_down"))) return e;

    // the y slots are strided by units x kUnitTokens rows; the grid's y index is the token
    dim3 cgrid((a.d + kCombineCols - 1) / kCombineCols, a.T);
    e = launch_pdl(mx_combine_kernel, cgrid, dim3(kCombineThreads), 0, s, static_cast<const float*>(m.y), m.umax,
                   kUnitTokens, a.d, a.wts, a.idx, static_cast<const int32_t*>(nullptr), a.E, a.k,
                   static_cast<const int32_t*>(m.rowmap), a.out, trace_stamp("combine"));
    trace_mark("combine", s);
    return e;
}

}  // namespace k3
