// MXFP4 repack / unpack between the compressed-tensors layout and ggml's
// 17-byte block (llama.cpp PR #26185 "model: add Kimi-K3 text model", review by
// GrEarl, section "repack_mxfp4_blocks is bit-exact - 0 mismatches over
// 11,010,048 values").
//
// Both layouts are flat over blocks: block g (= row * cols/32 + b) owns source
// bytes packed[16g .. 16g+15] and scale[g], and ggml bytes out[17g .. 17g+16].
// A CTA handles 256 consecutive blocks.  Source nibbles are read with 16-byte
// loads; the 17-byte blocks (not 16-byte aligned) are assembled in shared
// memory and written (or read) with 16-byte vector accesses over the CTA's
// contiguous 4352-byte span.  Integer work only; bit-exact.
#include "common.cuh"

namespace k3 {
namespace {

constexpr int kBlocksPerCta = 256;
constexpr int kSpan = kBlocksPerCta * 17;  // 4352 bytes, a multiple of 16

// 8 source bytes a (elements 0..15) and 8 bytes b (elements 16..31) of one
// block -> the 16 qs bytes: qs[2i] = lo(a_i) | lo(b_i) << 4,
// qs[2i+1] = hi(a_i) | hi(b_i) << 4.
__device__ __forceinline__ void to_qs(uint32_t a, uint32_t b, uint32_t& q0, uint32_t& q1) {
    uint32_t ev = (a & 0x0F0F0F0Fu) | ((b & 0x0F0F0F0Fu) << 4);
    uint32_t od = ((a >> 4) & 0x0F0F0F0Fu) | (b & 0xF0F0F0F0u);
    q0 = __byte_perm(ev, od, 0x5140);  // ev0 od0 ev1 od1
    q1 = __byte_perm(ev, od, 0x7362);  // ev2 od2 ev3 od3
}

// inverse: qs words -> source bytes
__device__ __forceinline__ void from_qs(uint32_t q0, uint32_t q1, uint32_t& a, uint32_t& b) {
    uint32_t ev = __byte_perm(q0, q1, 0x6420);  // qs[0], qs[2], qs[4], qs[6]
    uint32_t od = __byte_perm(q0, q1, 0x7531);  // qs[1], qs[3], qs[5], qs[7]
    a = (ev & 0x0F0F0F0Fu) | ((od & 0x0F0F0F0Fu) << 4);
    b = ((ev >> 4) & 0x0F0F0F0Fu) | (od & 0xF0F0F0F0u);
}

__global__ void __launch_bounds__(kBlocksPerCta)
repack_kernel(const uint8_t* __restrict__ packed, const uint8_t* __restrict__ scale,
              int64_t nblocks, uint8_t* __restrict__ out) {
    __shared__ __align__(16) uint8_t sm[kSpan];
    const int64_t g0 = static_cast<int64_t>(blockIdx.x) * kBlocksPerCta;
    const int64_t g = g0 + threadIdx.x;
    const int64_t left = nblocks - g0;
    const int nb = left < kBlocksPerCta ? static_cast<int>(left) : kBlocksPerCta;
    if (threadIdx.x < nb) {
        uint4 v = *reinterpret_cast<const uint4*>(packed + 16 * g);
        uint32_t q[4];
        to_qs(v.x, v.z, q[0], q[1]);  // bytes 0..3 with bytes 8..11
        to_qs(v.y, v.w, q[2], q[3]);  // bytes 4..7 with bytes 12..15
        uint8_t* dst = sm + 17 * threadIdx.x;
        dst[0] = scale[g];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
#pragma unroll
            for (int j = 0; j < 4; ++j) dst[1 + 4 * i + j] = static_cast<uint8_t>(q[i] >> (8 * j));
        }
    }
    __syncthreads();
    uint8_t* o = out + 17 * g0;
    const int bytes = 17 * nb;
    const bool vec = ((reinterpret_cast<uintptr_t>(o) & 15) == 0);
    if (vec) {
        const int nvec = bytes / 16;
        for (int i = threadIdx.x; i < nvec; i += blockDim.x)
            reinterpret_cast<uint4*>(o)[i] = reinterpret_cast<const uint4*>(sm)[i];
        for (int i = nvec * 16 + threadIdx.x; i < bytes; i += blockDim.x) o[i] = sm[i];
    } else {
        for (int i = threadIdx.x; i < bytes; i += blockDim.x) o[i] = sm[i];
    }
}

__global__ void __launch_bounds__(kBlocksPerCta)
unpack_kernel(const uint8_t* __restrict__ blocks, int64_t nblocks, uint8_t* __restrict__ packed,
              uint8_t* __restrict__ scale) {
    __shared__ __align__(16) uint8_t sm[kSpan];
    const int64_t g0 = static_cast<int64_t>(blockIdx.x) * kBlocksPerCta;
    const int64_t left = nblocks - g0;
    const int nb = left < kBlocksPerCta ? static_cast<int>(left) : kBlocksPerCta;
    const uint8_t* src = blocks + 17 * g0;
    const int bytes = 17 * nb;
    if ((reinterpret_cast<uintptr_t>(src) & 15) == 0) {
        const int nvec = bytes / 16;
        for (int i = threadIdx.x; i < nvec; i += blockDim.x)
            reinterpret_cast<uint4*>(sm)[i] = reinterpret_cast<const uint4*>(src)[i];
        for (int i = nvec * 16 + threadIdx.x; i < bytes; i += blockDim.x) sm[i] = src[i];
    } else {
        for (int i = threadIdx.x; i < bytes; i += blockDim.x) sm[i] = src[i];
    }
    __syncthreads();
    if (threadIdx.x < nb) {
        const int64_t g = g0 + threadIdx.x;
        const uint8_t* b = sm + 17 * threadIdx.x;
        uint32_t q[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            q[i] = b[1 + 4 * i] | (b[2 + 4 * i] << 8) | (b[3 + 4 * i] << 16) |
                   (static_cast<uint32_t>(b[4 + 4 * i]) << 24);
        uint4 v;
        from_qs(q[0], q[1], v.x, v.z);
        from_qs(q[2], q[3], v.y, v.w);
        *reinterpret_cast<uint4*>(packed + 16 * g) = v;
        scale[g] = b[0];
    }
}

}  // namespace

cudaError_t launch_repack(const uint8_t* packed, const uint8_t* scale, int64_t nblocks,
                          uint8_t* out, cudaStream_t s) {
    if (nblocks <= 0) return cudaSuccess;
    const int64_t grid = (nblocks + kBlocksPerCta - 1) / kBlocksPerCta;
    repack_kernel<<<static_cast<unsigned>(grid), kBlocksPerCta, 0, s>>>(packed, scale, nblocks,
                                                                         out);
    return cudaGetLastError();
}

cudaError_t launch_unpack(const uint8_t* blocks, int64_t nblocks, uint8_t* packed,
                          uint8_t* scale, cudaStream_t s) {
    if (nblocks <= 0) return cudaSuccess;
    const int64_t grid = (nblocks + kBlocksPerCta - 1) / kBlocksPerCta;
    unpack_kernel<<<static_cast<unsigned>(grid), kBlocksPerCta, 0, s>>>(blocks, nblocks, packed,
                                                                         scale);
    return cudaGetLastError();
}

}  // namespace k3
