/*
 * k3moe.h - C ABI of the latent routed-expert MoE layer over MXFP4 weights
 * (Kimi-K3 style), hand-written CUDA for sm_103a (GB300).
 *
 * Sources (web pages, cited by title and section):
 *   [PR26185]  llama.cpp PR #26185 "model: add Kimi-K3 text model"
 *     - opening post (pwilkin): latent MoE (routed experts run at the latent
 *       width) and the "situ" activation replacing SwiGLU;
 *     - review by GrEarl, section "Dry run: prepare_tensors() completes, all
 *       93 layers mapped, file type = 38": 896 experts, 16 used, sigmoid
 *       expert-score gating, exp_probs_b, ffn_routed_{down,up,norm};
 *     - review by GrEarl, section "repack_mxfp4_blocks is bit-exact - 0
 *       mismatches over 11,010,048 values": the MXFP4 source format, the ggml
 *       17-byte block and the repack.
 *   [PR573]   Lucebox PR #573 "feat(kimi-k3): add DSpark Q8 artifact and shared
 *       speculative runtime", section "DSpark acceptance-contract
 *       correction": RMS epsilon 1e-5; section "Runtime validation": SSD-routed
 *       experts behind an 8 GiB device expert cache.
 *   [K3-Stuff] the K3-Stuff model page, "llama-cpp-patches", change 2: the page
 *       cache as the hot-expert cache (lazy fault-in, LRU eviction).
 *
 * Conventions for every entry point:
 *   - Every pointer argument is DEVICE memory owned by the caller unless the
 *     entry point says "host".  The library allocates nothing in these calls
 *     (scratch lives in the caller's workspace) and keeps no pointer after
 *     the call returns.
 *   - Tensors are dense and row-major.  bf16 tensors are passed as uint16_t
 *     bit patterns, fp32 as float.  Every base pointer must be 16-byte
 *     aligned (K3MOE_ERR_ALIGN otherwise).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Work is enqueued asynchronously; nothing synchronises the
 *     host except k3moe_get_status and k3moe_forward_host.
 *   - Host-detectable errors (null pointer, bad shape, misalignment, small
 *     workspace) return before anything is launched.  Errors found on the
 *     device (a non-finite router logit, an expired bounded wait) are
 *     recorded in the workspace status word; read them with
 *     k3moe_get_status.  Outputs are unspecified after an error, but every
 *     kernel terminates.
 *   - Results are deterministic: the same inputs give bitwise identical
 *     outputs, run to run.
 */
#ifndef K3MOE_H
#define K3MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define K3MOE_ABI_VERSION 4

typedef enum k3moe_status {
    K3MOE_OK = 0,
    K3MOE_ERR_INVALID_ARG = 1,  /* null pointer, non-positive size */
    K3MOE_ERR_SHAPE = 2,        /* unsupported shape (cols % 32, k > E, k > 32, ...) */
    K3MOE_ERR_ALIGN = 3,        /* a base pointer is not 16-byte aligned */
    K3MOE_ERR_WORKSPACE = 4,    /* workspace smaller than required */
    K3MOE_ERR_CUDA = 5,         /* a CUDA runtime call failed (launch, copy, ...) */
    K3MOE_ERR_NONFINITE = 6,    /* device: a router logit was NaN or inf, or a bias was NaN */
    K3MOE_ERR_TIMEOUT = 7,      /* device: a bounded wait inside a kernel expired */
    K3MOE_ERR_UNSUPPORTED = 8   /* activation or path not available for the shape */
} k3moe_status;

/* Gated expert activation.  The pages name a "situ" activation that replaces
 * SwiGLU ([PR26185], opening post) but do not define it; it is a pluggable
 * epilogue, exercised as silu(g) * u with g = W1 x (gate) and u = W3 x (up). */
typedef enum k3moe_act {
    K3MOE_ACT_SILU_GATED = 0
} k3moe_act;

/* Expert-path selector.  AUTO picks BLOCK_SCALED for T <= 1024 and
 * BF16_DEQUANT otherwise; BLOCK_SCALED with T > 1024 returns
 * K3MOE_ERR_UNSUPPORTED.
 *   BLOCK_SCALED: block-scaled tcgen05 MMAs (kind::mxf4) streaming the
 *            selected experts' E2M1 codes by TMA, E8M0 scales applied by the
 *            tensor cores, activations as E2M1 terms (five per token up to 8
 *            tokens, four beyond: each term encodes what the previous ones
 *            left over, with its own E8M0 scale per 32 inputs); split over
 *            the SMs.  Up to 8 tokens every active expert takes all tokens;
 *            beyond that each expert's tokens are cut into units of at most
 *            16 and an expert's weights are streamed once per unit.  This is
 *            the block-scaled option of the layer's design; activations
 *            quantised once to MXFP8 (E4M3 elements) instead of E2M1 terms
 *            leave an output error of several percent of the row RMS, over
 *            the layer's bound, so they are not offered.
 *   BF16_DEQUANT: tcgen05 grouped GEMMs with in-shared-memory dequantisation
 *            of the MXFP4 weights to f16 (exact: an E2M1 value times a power
 *            of two within f16's range; same tensor-core rate as bf16),
 *            TMA-fed, TMEM accumulators; f16 token rows.
 * DECODE and GROUPED are the names of ABI version 3 for the same values. */
typedef enum k3moe_path {
    K3MOE_PATH_AUTO = 0,
    K3MOE_PATH_BLOCK_SCALED = 1,
    K3MOE_PATH_BF16_DEQUANT = 2,
    K3MOE_PATH_DECODE = K3MOE_PATH_BLOCK_SCALED,
    K3MOE_PATH_GROUPED = K3MOE_PATH_BF16_DEQUANT
} k3moe_path;

/* One MoE layer.  All pointers are device memory owned by the caller and must
 * stay valid while work that uses them is in flight.
 *
 * Expert weights ([PR26185], GrEarl, "repack_mxfp4_blocks is bit-exact"):
 * compressed-tensors MXFP4, logical [out, in] per expert, exactly as the
 * checkpoint stores each weight_packed / weight_scale pair.  `*_q` holds two
 * E2M1 codes per byte (element 2i in the low nibble, sign in bit 3,
 * magnitudes [0,.5,1,1.5,2,3,4,6]) and is 32-byte aligned; `*_s` holds one
 * E8M0 byte e per 32 consecutive inputs of a row (value 2^(e-127); e = 255,
 * NaN in the format, is not allowed), 16-byte aligned:
 *   w1_q [E, f, d/2]   w1_s [E, f, d/32]   gate projection
 *   w3_q [E, f, d/2]   w3_s [E, f, d/32]   up projection
 *   w2_q [E, d, f/2]   w2_s [E, d, f/32]   down projection
 * d and f are multiples of 64.  When d and f are multiples of 512 the kernels
 * read the scale rows as they are (a TMA box of 16 bytes x 128 rows per
 * 512-input stage, re-laid in shared memory); otherwise each forward first
 * rewrites all three scale arrays into the prepared layout in its workspace
 * (1/32 of the expert bytes, read and written once per call).
 * Optional fast path: w1_sf, w3_sf, w2_sf, the same scales in the prepared
 * layout that k3moe_prepare_scales writes (all three or none; NULL = use the
 * canonical arrays).  When given they are read instead of w*_s, which may
 * then be NULL.
 * Router ([PR26185], GrEarl, "Dry run"): logits l = x_r W_r^T, scores
 * s = sigmoid(l); the k experts with the largest s + b are selected (ties to
 * the lower index, slots listed in that order); combine weights are
 * s / sum(s) over the selected k (the bias only steers selection).
 * Block mode (D > 0): the input is h [T, D]; hn = RMSNorm(h) * gamma (eps),
 * the router reads hn (d_router = D), the experts read z = hn W_down^T
 * [T, d], and the output is W_up applied to the combined latent rows.
 *
 * Weight format (`format`):
 *   K3MOE_FORMAT_SPLIT (0): the codes and scales above.
 *   K3MOE_FORMAT_GGML  (1): llama.cpp's MXFP4 blocks, as k3moe_repack_mxfp4
 *     writes them ([PR26185], GrEarl, "repack_mxfp4_blocks is bit-exact"):
 *     w1_q [E, f, d/32, 17], w3_q [E, f, d/32, 17], w2_q [E, d, f/32, 17]
 *     (byte 0 of a block = the E8M0 byte e, bytes 1..16 = element j in the
 *     low and element j + 16 in the high nibble of byte j), 16-byte aligned;
 *     the scale pointers are unused (may be NULL).  The streaming kernels
 *     read the blocks as they are and convert them in shared memory; the
 *     result is bitwise that of the SPLIT format on the same weights.  d and
 *     f must be multiples of 512 (rows of whole 16-byte units); the
 *     BLOCK_SCALED path only (T <= 1024) and no expert cache (UNSUPPORTED
 *     otherwise). */
typedef enum k3moe_format {
    K3MOE_FORMAT_SPLIT = 0,
    K3MOE_FORMAT_GGML = 1
} k3moe_format;

typedef struct k3moe_layer_desc {
    int32_t E;          /* routed experts (896) */
    int32_t k;          /* experts per token (16), 1 <= k <= min(E, 32) */
    int32_t d;          /* latent width (3584), multiple of 64 */
    int32_t f;          /* expert hidden width (3072), multiple of 64 */
    int32_t d_router;   /* router input width: d (latent mode) or D (block mode) */
    int32_t act;        /* k3moe_act */
    int32_t path;       /* k3moe_path */
    int32_t D;          /* block mode: model width (7168), multiple of 128; 0 = latent mode */
    float eps;          /* block mode: RMSNorm epsilon (1e-5 per [PR573]) */
    int32_t format;     /* k3moe_format of the expert weights */
    const uint8_t* w1_q;
    const uint8_t* w3_q;
    const uint8_t* w2_q;
    const uint8_t* w1_s;         /* canonical E8M0 scales of w1 */
    const uint8_t* w3_s;         /* canonical E8M0 scales of w3 */
    const uint8_t* w2_s;         /* canonical E8M0 scales of w2 */
    const uint8_t* w1_sf;        /* optional: prepared scales of w1 (NULL = use w1_s) */
    const uint8_t* w3_sf;        /* optional: prepared scales of w3 */
    const uint8_t* w2_sf;        /* optional: prepared scales of w2 */
    const uint16_t* router_w;    /* [E, d_router] bf16 */
    const float* router_b;       /* [E] fp32 selection bias (exp_probs_b) */
    const uint16_t* norm_gamma;  /* block mode: [D] bf16 (ffn_routed_norm) */
    const uint16_t* w_down;      /* block mode: [d, D] bf16 (ffn_routed_down) */
    const uint16_t* w_up;        /* block mode: [D, d] bf16 (ffn_routed_up) */
} k3moe_layer_desc;

/* Library ABI version (K3MOE_ABI_VERSION of the build). */
int k3moe_abi_version(void);

/* Testing aid for the device-side failure path; the paper has no
 * counterpart.  k3moe_inject_fault(K3MOE_FAULT_DROP_SIGNAL) arms a fault for
 * the next k3moe_forward (eager, or the set-up forward of a graph creation)
 * issued by the calling host thread on the BLOCK_SCALED path: in the W1/W3
 * streaming kernel, the first CTA's producer never signals its first pipeline
 * stage, and every bounded wait of that launch gives up after 1 ms instead of
 * 2 s.  The MMA issuer waiting for that stage records K3MOE_ERR_TIMEOUT in the
 * workspace status word; the CTA's roles stop, its copies in flight land, its
 * tensor memory is released and the kernel returns; the rest of the forward
 * runs to its end and its output is unspecified.  No wait is left unbounded
 * and nothing faults.  0 disarms.  Returns the previously armed code.  The
 * next forward consumes the armed code whatever its path. */
#define K3MOE_FAULT_DROP_SIGNAL 1
int k3moe_inject_fault(int code);

/* Static description of a status code (never NULL). */
const char* k3moe_status_string(int status);

/* MXFP4 repack: compressed-tensors (packed, scale) -> ggml 17-byte blocks.
 * [PR26185], GrEarl, "repack_mxfp4_blocks is bit-exact": block b of a row is
 * byte 0 = e (stored unchanged; ggml decodes it as 2^(e-128) with doubled
 * kvalues, so the value is unchanged), bytes 1..16 = qs with element j in the
 * low nibble and element j+16 in the high nibble of qs[j].
 *   packed     [rows, cols/2] uint8 (device)
 *   scale      [rows, cols/32] uint8 (device)
 *   blocks_out [rows, cols/32, 17] uint8 (device; no alignment needed)
 * Errors: INVALID_ARG (null, rows or cols <= 0), SHAPE (cols % 32 != 0),
 * ALIGN (packed not 16-byte aligned), CUDA. Bit-exact integer work. */
k3moe_status k3moe_repack_mxfp4(const uint8_t* packed, const uint8_t* scale, int64_t rows,
                                int64_t cols, uint8_t* blocks_out, void* stream);

/* Inverse of k3moe_repack_mxfp4 (ggml blocks -> packed nibbles + E8M0).
 *   blocks [rows, cols/32, 17] uint8; packed_out [rows, cols/2] (16-byte
 *   aligned); scale_out [rows, cols/32].  Errors as for the repack. */
k3moe_status k3moe_unpack_mxfp4(const uint8_t* blocks, int64_t rows, int64_t cols,
                                uint8_t* packed_out, uint8_t* scale_out, void* stream);

/* Block-scale preparation for the tensor-core kernels (an optional fast
 * path: k3moe_forward also takes the canonical arrays).  The canonical E8M0
 * array of a weight matrix, E experts of `rows` rows with one byte per 32 of
 * the `cols` inputs, is regrouped per expert into 512-byte atoms, one per
 * tile of 128 rows and 128-wide input group (ceil(rows / 128) tiles and
 * ceil(cols / 128) groups per expert; rows past `rows` and blocks past
 * cols / 32 are zero): byte 16 (m % 32) + 4 (m / 32) + b of an atom holds row
 * m of the tile and block b of the group (the order in which tcgen05.cp
 * spreads scales over the TMEM lanes that the block-scaled MMA reads: row m
 * from lane m, column m / 32).  The atom of (expert, tile, group) starts at
 * byte ((e * tiles + tile) * groups + group) * 512.
 *   scale [E, rows, cols/32] uint8 (device)
 *   sf    k3moe_prepared_scales_size(E, rows, cols) bytes (device)
 * A byte permutation with zero padding: bit-exact, deterministic.  rows and
 * cols multiples of 64.  The paper stores scales row by row; the atoms are
 * this library's layout.  Errors: INVALID_ARG, SHAPE, ALIGN (16-byte), CUDA. */
size_t k3moe_prepared_scales_size(int64_t E, int64_t rows, int64_t cols);
k3moe_status k3moe_prepare_scales(const uint8_t* scale, int64_t E, int64_t rows, int64_t cols,
                                  uint8_t* sf, void* stream);

/* Inverse of k3moe_prepare_scales (prepared atoms -> canonical array; the
 * padding is not read). */
k3moe_status k3moe_unprepare_scales(const uint8_t* sf, int64_t E, int64_t rows, int64_t cols,
                                    uint8_t* scale, void* stream);

/* Workspace bytes that k3moe_route needs for T tokens and E experts. */
size_t k3moe_route_workspace_size(int32_t T, int32_t E);

/* Router: logits, sigmoid scores, biased top-k selection, renormalised
 * weights ([PR26185], GrEarl, "Dry run": sigmoid gating, exp_probs_b, top-16
 * of 896).
 *   x        [T, d_r] bf16       router input
 *   router_w [E, d_r] bf16
 *   bias     [E] fp32
 *   idx_out  [T, k] int32        selected experts, slot order = (s+b) desc, index asc
 *   w_out    [T, k] fp32         s / sum(s) over the selected experts
 *   logits_out [T, E] fp32 or NULL  the fp32 logits the selection used
 *   ws, ws_bytes                 scratch >= k3moe_route_workspace_size(T, E)
 * Logits accumulate bf16 products in fp32; s = 1 / (1 + expf(-l)) and
 * s + b are fp32.  Errors: INVALID_ARG, SHAPE (k > 32, k > E, E > 1024,
 * d_r not a multiple of 64), ALIGN, WORKSPACE, CUDA; device: NONFINITE (a
 * logit was not finite). */
k3moe_status k3moe_route(const uint16_t* x, int32_t T, int32_t d_r, const uint16_t* router_w,
                         const float* bias, int32_t E, int32_t k, int32_t* idx_out,
                         float* w_out, float* logits_out, void* ws, size_t ws_bytes,
                         void* stream);

/* k3moe_route without a workspace, for callers that cannot allocate device
 * memory or hand the library a scratch buffer: code whose device memory must
 * all come from a framework-owned pool, or a latency-critical decode loop in
 * which cudaMalloc (which can synchronise the whole device) is not allowed.
 * The paper has no counterpart: this is an integration convenience of this
 * library, computing exactly what k3moe_route computes (same kernel).
 *
 * Scratch: a file-scope device array of 33,024 bytes (a 256-byte header plus
 * room for 8 x 1024 fp32 logits), part of the library's module image, so every
 * GPU that loads the library holds it until the process exits.  Limits:
 * T <= 8 and E <= 1024; larger sizes return K3MOE_ERR_SHAPE (use k3moe_route
 * with a workspace).  No cudaMalloc, cudaFree or other allocation happens in
 * the call.
 *
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current) and caches it for the
 * life of the process; make that first call before any stream capture.  The
 * cached address belongs to the device's current context: after
 * cudaDeviceReset on that device, do not call this entry point again in the
 * same process.  Every call shares the array and it
 * keeps the last call's contents: each call clears the header on `stream`
 * before its kernel, and calls whose work overlaps on the GPU (different
 * streams, or different host threads) race on it, so order them.  Device-side
 * errors (a non-finite logit) are not reported by this entry point.
 * Arguments, layouts and the other errors are those of k3moe_route. */
k3moe_status k3moe_route_noalloc(const uint16_t* x, int32_t T, int32_t d_r,
                                 const uint16_t* router_w, const float* bias, int32_t E,
                                 int32_t k, int32_t* idx_out, float* w_out, float* logits_out,
                                 void* stream);

/* Expert histogram, exclusive scan and token permutation of a selection.
 * Pairs are numbered p = t*k + j.
 *   idx      [T, k] int32 in [0, E)
 *   counts   [E] int32; offsets [E+1] int32 (exclusive scan, offsets[E] = T*k)
 *   perm     [T*k] int32: row r of the permuted order holds pair perm[r];
 *            rows of expert e are offsets[e]..offsets[e+1]-1, tokens ascending
 *   inv      [T*k] int32: inv[p] = row of pair p
 * Scratch: ws of k3moe_route_workspace_size(T, E) bytes.  Integer work,
 * deterministic.  Errors: INVALID_ARG, SHAPE, ALIGN, WORKSPACE, CUDA. */
k3moe_status k3moe_permute(const int32_t* idx, int32_t T, int32_t k, int32_t E, int32_t* counts,
                           int32_t* offsets, int32_t* perm, int32_t* inv, void* ws,
                           size_t ws_bytes, void* stream);

/* RMSNorm over rows ([PR26185] ffn_routed_norm; eps 1e-5 per [PR573]):
 * out = bf16(h / sqrt(mean(h^2) + eps) * gamma), fp32 arithmetic.
 *   h [T, D] bf16, gamma [D] bf16, out [T, D] bf16.  D % 8 == 0. */
k3moe_status k3moe_rmsnorm(const uint16_t* h, int32_t T, int32_t D, const uint16_t* gamma,
                           float eps, uint16_t* out, void* stream);

/* Dense bf16 GEMM on tcgen05 (the latent projections ffn_routed_down/up and
 * the router logits at large T): out[t, n] = sum_c x[t, c] * w[n, c].
 *   x [T, K] bf16, w [N, K] bf16, out [T, N] bf16 (out_fp32 = 0) or fp32 (1).
 *   N % 128 == 0, K % 64 == 0, T >= 1.  fp32 accumulation in tensor memory. */
k3moe_status k3moe_gemm_bf16(const uint16_t* x, const uint16_t* w, int32_t T, int32_t N,
                             int32_t K, void* out, int32_t out_fp32, void* stream);

/* Workspace bytes that k3moe_forward needs for up to T_max tokens.  A new
 * workspace must be zero-filled once before its first use (cudaMemset); the
 * library keeps its 256-byte header consistent from then on.  The same holds
 * for the workspaces of k3moe_route and k3moe_permute. */
size_t k3moe_workspace_size(const k3moe_layer_desc* desc, int32_t T_max);

/* The MoE layer (latent mode) or the full latent block (block mode).
 *   hidden [T, d] bf16 (latent mode) or [T, D] bf16 (block mode)
 *   out    same shape as hidden, bf16
 *   ws     scratch of at least k3moe_workspace_size(desc, T) bytes
 * out[t] = sum_j w[t,j] * W2_e (act(W1_e x_t, W3_e x_t)), e = idx[t,j].
 * Both paths stage each (token, expert) result in fp32 and sum a token's
 * k terms in slot order, so the result does not depend on scheduling.
 * Errors: INVALID_ARG, SHAPE, ALIGN, WORKSPACE, UNSUPPORTED, CUDA; device
 * errors via k3moe_get_status. */
k3moe_status k3moe_forward(const k3moe_layer_desc* desc, const uint16_t* hidden, int32_t T,
                           uint16_t* out, void* ws, size_t ws_bytes, void* stream);

/* The experts and the combine of the layer on a selection the caller made
 * (latent mode): no router runs; out[t] = sum_j wts[t,j] * expert_{idx[t,j]}(
 * hidden[t]), summed in slot order, the expert path as k3moe_forward picks
 * it.  For expert parallelism ([PR26185]: the pages place expert stacks
 * across devices): a rank that holds experts [r E_l, (r + 1) E_l) runs this
 * with a descriptor of its E_l experts, k = 1 and the rows other ranks sent
 * it, each with the local index of its expert and its combine weight.
 *   hidden [T, d] bf16, idx [T, k] int32 in [0, E), wts [T, k] fp32 (device),
 *   out [T, d] bf16; ws as for k3moe_forward (k3moe_workspace_size).
 * Errors: those of k3moe_forward; UNSUPPORTED in block mode; device:
 * INVALID_ARG if an index is outside [0, E) (the output is then undefined). */
k3moe_status k3moe_forward_routed(const k3moe_layer_desc* desc, const uint16_t* hidden, int32_t T,
                                  const int32_t* idx, const float* wts, uint16_t* out, void* ws,
                                  size_t ws_bytes, void* stream);

/* k3moe_forward on HOST buffers: copies hidden (host) to the device on
 * `stream`, runs the layer, copies out back to host memory and waits for the
 * stream.  Pinned host memory gives asynchronous copies; pageable memory
 * works too.  The workspace must hold k3moe_workspace_size(desc, T) plus
 * k3moe_host_staging_size(desc, T) bytes; the copies go through staging
 * buffers at fixed offsets of it.  The first call with a given descriptor
 * (its contents), workspace, size, T, stream and device runs the forward
 * directly and records it into a CUDA graph (host and driver objects, no
 * device memory); a later call with the same arguments replays that graph.
 * When the batch is at most 1 MiB (T * width * 2 bytes) the graph also holds
 * the two copies, from and to two page-locked host buffers of that size that
 * the library allocates with it: a replay then copies hidden into one with
 * memcpy, launches the graph, waits and copies the other into out_host.
 * The library keeps the 8 most recently used such graphs for the life of the
 * process.  A graph reads the buffers the descriptor points to, so weights
 * rewritten in place are seen; point the descriptor at new buffers (a new
 * key) rather than freeing and reallocating under an unchanged descriptor
 * with other shapes.  While tracing is on, or when `stream` is being
 * captured, every call runs directly. */
size_t k3moe_host_staging_size(const k3moe_layer_desc* desc, int32_t T);
k3moe_status k3moe_forward_host(const k3moe_layer_desc* desc, const uint16_t* hidden_host,
                                int32_t T, uint16_t* out_host, void* ws, size_t ws_bytes,
                                void* stream);

/* CUDA graph of one k3moe_forward with fixed buffers, for callers that run
 * the same layer call repeatedly (a decode loop): the graph replays every
 * kernel of the forward back to back on the device, without per-kernel host
 * launch overhead.  k3moe_graph_create waits for the device to be idle
 * (cudaDeviceSynchronize: earlier work on any stream may use the same
 * workspace or cache; no stream of the process may be capturing in global
 * capture mode during the call, since that synchronisation would be refused
 * and would invalidate that capture), runs the forward once on a private
 * stream (one-time set-up), then captures it (thread-local capture mode) and
 * instantiates the executable graph; it allocates the graph objects (host and
 * driver), which k3moe_graph_destroy frees.  The buffers named here must stay
 * valid while the graph exists; new inputs are written into `hidden` in place.
 * k3moe_graph_launch enqueues one replay on `stream` and allocates nothing.
 * Errors: those of k3moe_forward, CUDA if capture or instantiation fails. */
k3moe_status k3moe_graph_create(const k3moe_layer_desc* desc, const uint16_t* hidden, int32_t T,
                                uint16_t* out, void* ws, size_t ws_bytes, void** graph_out);
k3moe_status k3moe_graph_launch(void* graph, void* stream);
k3moe_status k3moe_graph_destroy(void* graph);

/* Host-resident experts behind a device expert cache.
 *
 * [K3-Stuff] (the K3-Stuff model page, "llama-cpp-patches", change 2) runs
 * the model with its experts outside device memory: the page cache is the
 * hot-expert cache, filled lazily and evicted least recently used; [PR573]
 * ("Runtime validation") does the same with an 8 GiB device expert cache and
 * batched verification routed per batch.  Here the six expert arrays of the
 * layer stay in HOST memory and `slots` experts at a time live in device
 * memory.  Each k3moe_forward_cached call, after routing, refreshes the
 * stamps of the used experts that are resident (hits), gives each missing
 * expert the least recently used slot that the call does not use (never-used
 * slots first; equal stamps: lower slot first; the i-th missing expert in
 * ascending index takes the i-th victim in ascending slot order), copies the
 * missing experts' codes and scale atoms from host memory into their slots on
 * the device (every SM reads the host arrays directly; on GB300 over
 * NVLink-C2C), and then runs the expert kernels on the slots.  Every token of
 * the call shares the fetch: an expert is fetched at most once per call (the
 * union of the call's selections, as in a batch of draft tokens).  The result
 * is bitwise the result of k3moe_forward on device-resident weights.
 *
 * All cache pointers are device memory owned by the caller:
 *   w1_q  [slots, f, d/2]   w3_q [slots, f, d/2]   w2_q [slots, d, f/2]
 *         (32-byte aligned)
 *   w1_s, w3_s, w2_s        the slots' scales, in the layout the layer
 *                           descriptor's scales use: canonical rows
 *                           ([slots, f, d/32], [slots, d, f/32]; d and f
 *                           multiples of 512) or, when the descriptor gives
 *                           prepared scales, k3moe_prepared_scales_size(slots,
 *                           f, d) bytes each
 *   state                   bookkeeping, k3moe_cache_state_size(E, slots)
 *                           bytes, set up by k3moe_cache_init before first use
 * min(E, T*k) <= slots <= E for every call (K3MOE_ERR_SHAPE otherwise). */
typedef struct k3moe_expert_cache {
    int32_t slots;      /* experts the device holds at a time */
    int32_t reserved;   /* must be 0 */
    uint8_t* w1_q;
    uint8_t* w3_q;
    uint8_t* w2_q;
    uint8_t* w1_s;
    uint8_t* w3_s;
    uint8_t* w2_s;
    void* state;
} k3moe_expert_cache;

/* Device bytes of the cache bookkeeping (a 256-byte header, the expert ->
 * slot map and per-slot arrays); 0 for non-positive sizes. */
size_t k3moe_cache_state_size(int32_t E, int32_t slots);

/* Marks every slot empty and clears the counters (on `stream`).
 * Errors: INVALID_ARG, SHAPE (slots > E or E > 1024), ALIGN, CUDA. */
k3moe_status k3moe_cache_init(void* state, int32_t E, int32_t slots, void* stream);

/* k3moe_forward with the expert weights in host memory.  The descriptor's
 * codes and scales (the canonical w*_s, or the prepared w*_sf when given)
 * point to HOST arrays in the layouts k3moe_forward takes, page-locked and
 * mapped into the device address space (cudaHostAlloc, or cudaHostRegister
 * with mapping); every other pointer is device memory.  Canonical scales need
 * d and f multiples of 512 here.  The BLOCK_SCALED path only (T <= 1024).  The
 * call keeps the cache state between calls; calls sharing a cache must be
 * ordered on one stream.  Errors: those of k3moe_forward; INVALID_ARG (null
 * host array, or one that is not page-locked host memory by
 * cudaPointerGetAttributes, e.g. a device array; reserved != 0), SHAPE
 * (slots), UNSUPPORTED (the
 * BF16_DEQUANT path, canonical scales with d or f not a multiple of 512);
 * device: INVALID_ARG if the state was not initialised for (E, slots). */
k3moe_status k3moe_forward_cached(const k3moe_layer_desc* desc, const k3moe_expert_cache* cache,
                                  const uint16_t* hidden, int32_t T, uint16_t* out, void* ws,
                                  size_t ws_bytes, void* stream);

/* Counters of a cache since k3moe_cache_init: calls, expert hits and misses
 * (a used expert counts once per call), bytes fetched from host memory, and
 * the hits and misses of the last call.  Synchronises `stream`.
 * Errors: INVALID_ARG (null, state not initialised), CUDA. */
typedef struct k3moe_cache_stats {
    uint64_t calls, hits, misses, bytes;
    int32_t last_hits, last_misses;
} k3moe_cache_stats;
k3moe_status k3moe_cache_read_stats(const void* state, void* stream, k3moe_cache_stats* out);

/* k3moe_graph_create for k3moe_forward_cached: every replay routes, updates
 * the cache and fetches what is missing, like an eager call.  The set-up
 * forward counts as a call of the cache (the capture itself runs nothing). */
k3moe_status k3moe_graph_create_cached(const k3moe_layer_desc* desc, const k3moe_expert_cache* cache,
                                       const uint16_t* hidden, int32_t T, uint16_t* out, void* ws,
                                       size_t ws_bytes, void** graph_out);

/* Copy the routing of the last k3moe_forward that used `ws` (device to
 * device, on `stream`): idx_out [T, k] int32, w_out [T, k] fp32, logits_out
 * [T, E] fp32 or NULL. */
k3moe_status k3moe_forward_routing(const k3moe_layer_desc* desc, const void* ws, int32_t T,
                                   int32_t* idx_out, float* w_out, float* logits_out,
                                   void* stream);

/* Block mode: copy the intermediates of the last k3moe_forward that used
 * `ws` (device to device, on `stream`; any output may be NULL): hn_out [T, D]
 * bf16, the normalised hidden (the router's input); z_out [T, d] bf16, the
 * latent input of the experts (hn W_down^T); m_out [T, d] bf16, the combined
 * latent rows before the up-projection.  Errors: INVALID_ARG, UNSUPPORTED
 * (latent mode), CUDA. */
k3moe_status k3moe_forward_intermediates(const k3moe_layer_desc* desc, const void* ws, int32_t T,
                                         uint16_t* hn_out, uint16_t* z_out, uint16_t* m_out,
                                         void* stream);

/* Read and clear the device status word of a workspace.  Synchronises
 * `stream`; *device_status receives K3MOE_OK or the first device error code.
 * Returns CUDA if the stream reported an error. */
k3moe_status k3moe_get_status(void* ws, void* stream, int32_t* device_status);

/* Kernel tracing, off by default, process-wide and meant for one host thread.
 * k3moe_trace(mode) returns the previous mode; mode is a bit set:
 *   bit 0 (1): k3moe_forward records a CUDA event on its stream after each
 *     kernel it launches (a forward captured into a CUDA graph captures the
 *     records as external-event nodes, and each replay re-records them).
 *     k3moe_trace_read waits for the last event and fills up to `max` entries
 *     with the kernel names (static strings) and the milliseconds between
 *     consecutive events of the most recently traced forward, and returns the
 *     number of entries (0 if the events cannot be read).  The records sit
 *     between the kernels, so they also stop the next kernel from starting
 *     early (programmatic launch) and each interval carries launch latency.
 *   bit 1 (2): device stamps.  Each kernel of the forward records, in a
 *     1.5 KB area of the caller's workspace, the global timer when its first
 *     CTA passes its dependency wait and when its last CTA finishes (the
 *     area is reset at the start of every forward, graph replays included).
 *     Nothing is inserted between the kernels, so the timeline is that of the
 *     untraced forward.  k3moe_trace_read_stamps synchronises the device,
 *     reads the stamps of the most recently stamped forward (its workspace
 *     must still exist) and fills up to `max` entries with the kernel names
 *     and the start and end in microseconds after the earliest start (-1 for
 *     a kernel that did not run); it returns the number of entries. */
int k3moe_trace(int mode);
int k3moe_trace_read(int max, const char** names, float* ms);
int k3moe_trace_read_stamps(int max, const char** names, double* start_us, double* end_us);

#ifdef __cplusplus
}
#endif

#endif /* K3MOE_H */
