// Host side of the k3moe C ABI: argument checks, workspace layout, dispatch.
// Every step of the layer runs in the kernels of this library; nothing here
// computes on the host.
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "common.cuh"

using namespace k3;

namespace {

constexpr int kDecodeMaxT = 8;
// the block-scaled streaming kernels also take up to this many tokens, grouped
// in units of at most 16 tokens of one expert (beyond it the experts see many
// tokens each and the grouped GEMMs are the better fit)
constexpr int kStreamMaxT = 1024;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned32(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }

int device_sms() {
    static std::mutex mu;
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev] == 0) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        cache[dev] = n > 0 ? n : 148;
    }
    return cache[dev];
}

// K3MOE_DEBUG=1 in the environment prints the CUDA error behind a
// K3MOE_ERR_CUDA status to stderr (read once)
bool debug_on() {
    static const bool on = [] {
        const char* v = getenv("K3MOE_DEBUG");
        return v && v[0] && v[0] != '0';
    }();
    return on;
}

k3moe_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return K3MOE_OK;
    if (debug_on()) fprintf(stderr, "k3moe: CUDA error %d (%s)\n", static_cast<int>(e), cudaGetErrorString(e));
    return K3MOE_ERR_CUDA;
}

// fault armed by k3moe_inject_fault for the next forward of this host thread
thread_local int g_inject = 0;

// PDL is on unless K3MOE_NO_PDL is set in the environment (read once)
bool pdl_on() {
    static const bool on = [] {
        const char* v = getenv("K3MOE_NO_PDL");
        return !(v && v[0] && v[0] != '0');
    }();
    return on;
}

// ---------------------------------------------------------------------------
// workspace layouts
// ---------------------------------------------------------------------------
struct Carve {
    size_t off = sizeof(WsHeader);
    size_t take(size_t bytes) {
        const size_t o = off;
        off = align_up(off + bytes);
        return o;
    }
};

struct RoutePlan {
    size_t logits, chunk, active, total;
};

RoutePlan route_plan(int T, int E) {
    Carve c;
    RoutePlan p;
    p.logits = c.take(static_cast<size_t>(T) * E * 4);
    p.chunk = c.take(permute_scratch_bytes(T, E));
    p.active = c.take(static_cast<size_t>(E + 1) * 4);
    p.total = c.off;
    return p;
}

// Which scales the expert kernels read: the caller's prepared atoms, the
// caller's canonical rows (d and f multiples of 512), or atoms that the
// forward writes into its workspace from the canonical rows first.
enum ScaleSource { SCALES_PREPARED = 0, SCALES_CANON = 1, SCALES_CANON_PREP = 2 };

ScaleSource scale_source(const k3moe_layer_desc* d) {
    if (d->w1_sf && d->w3_sf && d->w2_sf) return SCALES_PREPARED;
    return (d->d % 512 == 0 && d->f % 512 == 0) ? SCALES_CANON : SCALES_CANON_PREP;
}

struct FwdPlan {
    size_t stamps;                                  // device timeline (k3moe_trace mode 2)
    size_t sf1, sf3, sf2;                           // atoms written per call (SCALES_CANON_PREP)
    size_t logits, idx, wts, counts, offsets, active, perm, inv, chunk;
    size_t dec, y;                                  // decode scratch, shared y (fp32)
    size_t units;                                   // unit-grouped streaming scratch
    size_t xp, xp_exp, hb, h_amax, hp, hp_exp, tiles;  // grouped
    size_t hn, z, m;                                // block mode
    size_t total;
    int tiles_cap;
};

FwdPlan fwd_plan(const k3moe_layer_desc* d, int T) {
    Carve c;
    FwdPlan p{};
    const size_t P = static_cast<size_t>(T) * d->k;
    p.stamps = c.take(2 * kStampSlots * sizeof(uint64_t));
    if (d->format == K3MOE_FORMAT_SPLIT && scale_source(d) == SCALES_CANON_PREP) {
        p.sf1 = c.take(prepared_sf_bytes(d->E, d->f, d->d));
        p.sf3 = c.take(prepared_sf_bytes(d->E, d->f, d->d));
        p.sf2 = c.take(prepared_sf_bytes(d->E, d->d, d->f));
    }
    p.logits = c.take(static_cast<size_t>(T) * d->E * 4);
    p.idx = c.take(P * 4);
    p.wts = c.take(P * 4);
    p.counts = c.take(static_cast<size_t>(d->E) * 4);
    p.offsets = c.take(static_cast<size_t>(d->E + 1) * 4);
    p.active = c.take(static_cast<size_t>(d->E + 1) * 4);
    p.perm = c.take(P * 4);
    p.inv = c.take(P * 4);
    p.chunk = c.take(permute_scratch_bytes(T, d->E));
    const int Td = std::min(T, kDecodeMaxT);
    p.dec = c.take(mx_decode_scratch_bytes(Td, d->E, d->k, d->d, d->f));
    if (T > kDecodeMaxT && T <= kStreamMaxT) p.units = c.take(mx_units_scratch_bytes(T, d->E, d->k, d->d, d->f));
    p.y = c.take(P * d->d * 4);  // grouped path
    p.xp = c.take(P * d->d * 2);
    p.xp_exp = c.take(P * 4);
    p.hb = c.take(P * d->f * 4);
    p.h_amax = c.take(P * 4);
    p.hp = c.take(P * d->f * 2);
    p.hp_exp = c.take(P * 4);
    p.tiles_cap = static_cast<int>(grouped_tile_cap(T, d->E, d->k, d->d, d->f));
    p.tiles = c.take(2 * (static_cast<size_t>(p.tiles_cap) + 1) * 16);
    if (d->D > 0) {
        p.hn = c.take(static_cast<size_t>(T) * d->D * 2);
        p.z = c.take(static_cast<size_t>(T) * d->d * 2);
        p.m = c.take(static_cast<size_t>(T) * d->d * 2);
    }
    p.total = c.off;
    return p;
}

k3moe_status check_desc(const k3moe_layer_desc* d) {
    if (!d) return K3MOE_ERR_INVALID_ARG;
    if (d->E < 1 || d->k < 1 || d->d < 1 || d->f < 1 || d->d_router < 1) return K3MOE_ERR_INVALID_ARG;
    if (d->format != K3MOE_FORMAT_SPLIT && d->format != K3MOE_FORMAT_GGML) return K3MOE_ERR_INVALID_ARG;
    if (d->k > d->E || d->k > 32 || d->E > 1024) return K3MOE_ERR_SHAPE;
    if (d->d % 64 || d->f % 64) return K3MOE_ERR_SHAPE;  // the MMAs take 64 inputs at a time
    if (d->D < 0) return K3MOE_ERR_SHAPE;
    if (d->D > 0) {
        if (d->D % 128 || d->d % 128 || d->d_router != d->D) return K3MOE_ERR_SHAPE;
        if (!(d->eps >= 0.0f)) return K3MOE_ERR_INVALID_ARG;
        if (!d->norm_gamma || !d->w_down || !d->w_up) return K3MOE_ERR_INVALID_ARG;
        if (!aligned16(d->norm_gamma) || !aligned16(d->w_down) || !aligned16(d->w_up))
            return K3MOE_ERR_ALIGN;
    } else if (d->d_router != d->d) {
        return K3MOE_ERR_SHAPE;
    }
    if (d->act != K3MOE_ACT_SILU_GATED) return K3MOE_ERR_UNSUPPORTED;
    if (d->path < K3MOE_PATH_AUTO || d->path > K3MOE_PATH_BF16_DEQUANT) return K3MOE_ERR_INVALID_ARG;
    const bool ggml = d->format == K3MOE_FORMAT_GGML;
    const void* ptrs[] = {d->w1_q, d->w3_q, d->w2_q, d->router_w, d->router_b};
    for (const void* q : ptrs) {
        if (!q) return K3MOE_ERR_INVALID_ARG;
        if (!aligned16(q)) return K3MOE_ERR_ALIGN;
    }
    if (!ggml) {  // ggml blocks carry their scales
        // prepared scales: all three or none; without them the canonical arrays
        const int nsf = (d->w1_sf != nullptr) + (d->w3_sf != nullptr) + (d->w2_sf != nullptr);
        if (nsf != 0 && nsf != 3) return K3MOE_ERR_INVALID_ARG;
        const void* sc[] = {d->w1_sf, d->w3_sf, d->w2_sf};
        const void* cs[] = {d->w1_s, d->w3_s, d->w2_s};
        for (const void* q : nsf ? sc : cs) {
            if (!q) return K3MOE_ERR_INVALID_ARG;
            if (!aligned16(q)) return K3MOE_ERR_ALIGN;
        }
    }
    if (ggml) {
        // rows of d/32 (f/32) 17-byte blocks are whole 16-byte units for TMA
        if (d->d % 512 || d->f % 512) return K3MOE_ERR_SHAPE;
        return K3MOE_OK;
    }
    // E2M1 codes are read by TMA in 16-byte slots: 32-byte aligned bases
    if (!aligned32(d->w1_q) || !aligned32(d->w3_q) || !aligned32(d->w2_q)) return K3MOE_ERR_ALIGN;
    return K3MOE_OK;
}

// ---------------------------------------------------------------------------
// tracing: events between the kernel launches of one forward (mode bit 0),
// device stamps of each launch's first CTA start and last CTA end (bit 1)
// ---------------------------------------------------------------------------
struct Trace {
    std::mutex mu;
    int mode = 0;
    int n = 0;
    cudaEvent_t ev[33] = {};
    const char* names[32] = {};
    int n_last = 0;
    float ms_last[32] = {};
    const char* names_last[32] = {};
    uint64_t* stamp_base = nullptr;        // stamp area of the forward being issued
    int ns = 0;
    const char* snames[kStampSlots] = {};
    const uint64_t* stamp_last = nullptr;  // stamp area of the last stamped forward
    int ns_last = 0;
    const char* snames_last[kStampSlots] = {};
};
Trace g_trace;

// Inside a stream capture a plain event record is only a dependency of the
// capture; an external record becomes a node that records the event each
// time the graph runs, so its timing can be read afterwards.
void trace_record(cudaEvent_t ev, cudaStream_t s) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
        cudaEventRecordWithFlags(ev, s, cudaEventRecordExternal);
    else
        cudaEventRecord(ev, s);
}

void trace_begin(cudaStream_t s, uint64_t* stamps) {
    g_trace.stamp_base = nullptr;
    if (g_trace.mode & 1) {
        g_trace.n = 0;
        if (!g_trace.ev[0])
            for (auto& e : g_trace.ev) cudaEventCreate(&e);
        trace_record(g_trace.ev[0], s);
    }
    if ((g_trace.mode & 2) && stamps) {
        // starts at the largest value (atomicMin), ends at 0 (atomicMax); in a
        // captured forward these are memset nodes, so every replay starts clean
        cudaMemsetAsync(stamps, 0xFF, kStampSlots * sizeof(uint64_t), s);
        cudaMemsetAsync(stamps + kStampSlots, 0, kStampSlots * sizeof(uint64_t), s);
        g_trace.stamp_base = stamps;
        g_trace.ns = 0;
    }
}

void trace_end() {
    // the events are read in k3moe_trace_read (they may also be replayed by a
    // CUDA graph that captured this forward); remember the names now
    if (g_trace.mode & 1) {
        for (int i = 0; i < g_trace.n; ++i) g_trace.names_last[i] = g_trace.names[i];
        g_trace.n_last = g_trace.n;
    }
    if (g_trace.stamp_base) {
        for (int i = 0; i < g_trace.ns; ++i) g_trace.snames_last[i] = g_trace.snames[i];
        g_trace.ns_last = g_trace.ns;
        g_trace.stamp_last = g_trace.stamp_base;
        g_trace.stamp_base = nullptr;
    }
}

}  // namespace

namespace k3 {
bool pdl_enabled() { return pdl_on(); }

void trace_mark(const char* name, cudaStream_t s) {
    if (!(g_trace.mode & 1) || g_trace.n >= 32) return;
    g_trace.names[g_trace.n] = name;
    trace_record(g_trace.ev[g_trace.n + 1], s);
    ++g_trace.n;
}

uint64_t* trace_stamp(const char* name) {
    if (!g_trace.stamp_base || g_trace.ns >= kStampSlots) return nullptr;
    g_trace.snames[g_trace.ns] = name;
    return g_trace.stamp_base + g_trace.ns++;
}
}  // namespace k3

extern "C" {

int k3moe_trace(int enable) {
    std::lock_guard<std::mutex> lock(g_trace.mu);
    const int prev = g_trace.mode;
    g_trace.mode = enable & 3;
    return prev;
}

int k3moe_trace_read(int max, const char** names, float* ms) {
    std::lock_guard<std::mutex> lock(g_trace.mu);
    if (g_trace.n_last > 0) {
        const int n = g_trace.n_last;
        if (cudaEventSynchronize(g_trace.ev[n]) != cudaSuccess) {
            cudaGetLastError();  // leave no pending error behind
            return 0;
        }
        for (int i = 0; i < n; ++i) {
            float t = 0.0f;
            if (cudaEventElapsedTime(&t, g_trace.ev[i], g_trace.ev[i + 1]) != cudaSuccess) {
                cudaGetLastError();
                return 0;
            }
            g_trace.ms_last[i] = t;
        }
    }
    const int n = g_trace.n_last < max ? g_trace.n_last : max;
    for (int i = 0; i < n; ++i) {
        if (names) names[i] = g_trace.names_last[i];
        if (ms) ms[i] = g_trace.ms_last[i];
    }
    return n;
}

int k3moe_trace_read_stamps(int max, const char** names, double* start_us, double* end_us) {
    std::lock_guard<std::mutex> lock(g_trace.mu);
    const int n = g_trace.ns_last < max ? g_trace.ns_last : max;
    if (n <= 0 || !g_trace.stamp_last) return 0;
    uint64_t st[2 * kStampSlots];
    if (cudaDeviceSynchronize() != cudaSuccess ||
        cudaMemcpy(st, g_trace.stamp_last, sizeof(st), cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    uint64_t t0 = ~0ull;
    for (int i = 0; i < n; ++i) t0 = st[i] < t0 ? st[i] : t0;
    for (int i = 0; i < n; ++i) {
        const bool ran = st[i] != ~0ull && st[kStampSlots + i] >= st[i];
        if (names) names[i] = g_trace.snames_last[i];
        if (start_us) start_us[i] = ran ? (st[i] - t0) * 1e-3 : -1.0;
        if (end_us) end_us[i] = ran ? (st[kStampSlots + i] - t0) * 1e-3 : -1.0;
    }
    return n;
}

int k3moe_abi_version(void) { return K3MOE_ABI_VERSION; }

int k3moe_inject_fault(int code) {
    const int prev = g_inject;
    g_inject = code == K3MOE_FAULT_DROP_SIGNAL ? code : 0;
    return prev;
}

const char* k3moe_status_string(int status) {
    switch (status) {
        case K3MOE_OK: return "ok";
        case K3MOE_ERR_INVALID_ARG: return "invalid argument";
        case K3MOE_ERR_SHAPE: return "unsupported shape";
        case K3MOE_ERR_ALIGN: return "pointer not 16-byte aligned";
        case K3MOE_ERR_WORKSPACE: return "workspace too small";
        case K3MOE_ERR_CUDA: return "CUDA error";
        case K3MOE_ERR_NONFINITE: return "non-finite router logit";
        case K3MOE_ERR_TIMEOUT: return "bounded wait expired on the device";
        case K3MOE_ERR_UNSUPPORTED: return "unsupported activation or path";
        default: return "unknown status";
    }
}

k3moe_status k3moe_repack_mxfp4(const uint8_t* packed, const uint8_t* scale, int64_t rows,
                                int64_t cols, uint8_t* blocks_out, void* stream) {
    if (!packed || !scale || !blocks_out || rows <= 0 || cols <= 0) return K3MOE_ERR_INVALID_ARG;
    if (cols % 32) return K3MOE_ERR_SHAPE;
    if (!aligned16(packed)) return K3MOE_ERR_ALIGN;
    return cuda_status(launch_repack(packed, scale, rows * (cols / 32), blocks_out,
                                     static_cast<cudaStream_t>(stream)));
}

k3moe_status k3moe_unpack_mxfp4(const uint8_t* blocks, int64_t rows, int64_t cols,
                                uint8_t* packed_out, uint8_t* scale_out, void* stream) {
    if (!blocks || !packed_out || !scale_out || rows <= 0 || cols <= 0) return K3MOE_ERR_INVALID_ARG;
    if (cols % 32) return K3MOE_ERR_SHAPE;
    if (!aligned16(packed_out)) return K3MOE_ERR_ALIGN;
    return cuda_status(launch_unpack(blocks, rows * (cols / 32), packed_out, scale_out,
                                     static_cast<cudaStream_t>(stream)));
}

size_t k3moe_prepared_scales_size(int64_t E, int64_t rows, int64_t cols) {
    if (E < 1 || rows < 1 || cols < 1 || rows > (1 << 30) || cols > (1 << 30)) return 0;
    return prepared_sf_bytes(E, static_cast<int>(rows), static_cast<int>(cols));
}

namespace {
k3moe_status check_prepare(const void* a, const void* b, int64_t E, int64_t rows, int64_t cols) {
    if (!a || !b || E < 1 || rows < 1 || cols < 1) return K3MOE_ERR_INVALID_ARG;
    if (rows % 64 || cols % 64 || rows > (1 << 30) || cols > (1 << 30)) return K3MOE_ERR_SHAPE;
    if (!aligned16(a) || !aligned16(b)) return K3MOE_ERR_ALIGN;
    return K3MOE_OK;
}
}  // namespace

k3moe_status k3moe_prepare_scales(const uint8_t* scale, int64_t E, int64_t rows, int64_t cols, uint8_t* sf,
                                  void* stream) {
    const k3moe_status st = check_prepare(scale, sf, E, rows, cols);
    if (st != K3MOE_OK) return st;
    return cuda_status(launch_prepare_sf(scale, E, static_cast<int>(rows), static_cast<int>(cols), sf, 0,
                                         static_cast<cudaStream_t>(stream)));
}

k3moe_status k3moe_unprepare_scales(const uint8_t* sf, int64_t E, int64_t rows, int64_t cols, uint8_t* scale,
                                    void* stream) {
    const k3moe_status st = check_prepare(sf, scale, E, rows, cols);
    if (st != K3MOE_OK) return st;
    return cuda_status(launch_prepare_sf(scale, E, static_cast<int>(rows), static_cast<int>(cols),
                                         const_cast<uint8_t*>(sf), 1, static_cast<cudaStream_t>(stream)));
}

size_t k3moe_route_workspace_size(int32_t T, int32_t E) {
    if (T < 1 || E < 1) return 0;
    return route_plan(T, E).total;
}

k3moe_status k3moe_route(const uint16_t* x, int32_t T, int32_t d_r, const uint16_t* router_w,
                         const float* bias, int32_t E, int32_t k, int32_t* idx_out,
                         float* w_out, float* logits_out, void* ws, size_t ws_bytes,
                         void* stream) {
    if (!x || !router_w || !bias || !idx_out || !w_out || !ws) return K3MOE_ERR_INVALID_ARG;
    if (T < 1 || d_r < 1 || E < 1 || k < 1) return K3MOE_ERR_INVALID_ARG;
    if (k > E || k > 32 || E > 1024 || d_r % 64) return K3MOE_ERR_SHAPE;
    const void* ptrs[] = {x, router_w, bias, idx_out, w_out, ws};
    for (const void* p : ptrs)
        if (!aligned16(p)) return K3MOE_ERR_ALIGN;
    if (logits_out && !aligned16(logits_out)) return K3MOE_ERR_ALIGN;
    const RoutePlan p = route_plan(T, E);
    if (ws_bytes < p.total) return K3MOE_ERR_WORKSPACE;
    char* base = static_cast<char*>(ws);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    RouteArgs a{};
    a.x = x; a.T = T; a.d_r = d_r; a.w = router_w; a.bias = bias; a.E = E; a.k = k;
    a.idx = idx_out; a.wts = w_out;
    a.logits = logits_out ? logits_out : reinterpret_cast<float*>(base + p.logits);
    a.hdr = reinterpret_cast<WsHeader*>(base);
    if (T <= kDecodeMaxT) return cuda_status(launch_route_small(a, s));
    cudaError_t e = cudaSuccess;
    if (T >= 64 && E % 128 == 0) {
        e = launch_gemm_bf16(x, router_w, T, E, d_r, a.logits, 1, a.hdr, device_sms(), s, "router_logits");
        if (e == cudaErrorNotSupported) e = launch_logits_simt(a, s);
    } else {
        e = launch_logits_simt(a, s);
    }
    if (e != cudaSuccess) return K3MOE_ERR_CUDA;
    return cuda_status(launch_topk(a, s));
}

k3moe_status k3moe_route_noalloc(const uint16_t* x, int32_t T, int32_t d_r,
                                 const uint16_t* router_w, const float* bias, int32_t E,
                                 int32_t k, int32_t* idx_out, float* w_out, float* logits_out,
                                 void* stream) {
    if (!x || !router_w || !bias || !idx_out || !w_out) return K3MOE_ERR_INVALID_ARG;
    if (T < 1 || d_r < 1 || E < 1 || k < 1) return K3MOE_ERR_INVALID_ARG;
    if (T > kNoAllocMaxT || E > kNoAllocMaxE) return K3MOE_ERR_SHAPE;
    if (k > E || k > 32 || d_r % 64) return K3MOE_ERR_SHAPE;
    const void* ptrs[] = {x, router_w, bias, idx_out, w_out};
    for (const void* p : ptrs)
        if (!aligned16(p)) return K3MOE_ERR_ALIGN;
    if (logits_out && !aligned16(logits_out)) return K3MOE_ERR_ALIGN;
    RouteArgs a{};
    a.x = x; a.T = T; a.d_r = d_r; a.w = router_w; a.bias = bias; a.E = E; a.k = k;
    a.idx = idx_out; a.wts = w_out; a.logits = logits_out;
    return cuda_status(launch_route_noalloc(a, static_cast<cudaStream_t>(stream)));
}

k3moe_status k3moe_permute(const int32_t* idx, int32_t T, int32_t k, int32_t E, int32_t* counts,
                           int32_t* offsets, int32_t* perm, int32_t* inv, void* ws,
                           size_t ws_bytes, void* stream) {
    if (!idx || !counts || !offsets || !perm || !inv || !ws) return K3MOE_ERR_INVALID_ARG;
    if (T < 1 || k < 1 || E < 1) return K3MOE_ERR_INVALID_ARG;
    if (k > E || k > 32) return K3MOE_ERR_SHAPE;
    const void* ptrs[] = {idx, counts, offsets, perm, inv, ws};
    for (const void* p : ptrs)
        if (!aligned16(p)) return K3MOE_ERR_ALIGN;
    const RoutePlan p = route_plan(T, E);
    if (ws_bytes < p.total) return K3MOE_ERR_WORKSPACE;
    char* base = static_cast<char*>(ws);
    return cuda_status(launch_permute(idx, T, k, E, counts, offsets, perm, inv,
                                      reinterpret_cast<int32_t*>(base + p.active),
                                      base + p.chunk, reinterpret_cast<WsHeader*>(base),
                                      static_cast<cudaStream_t>(stream)));
}

k3moe_status k3moe_rmsnorm(const uint16_t* h, int32_t T, int32_t D, const uint16_t* gamma,
                           float eps, uint16_t* out, void* stream) {
    if (!h || !gamma || !out || T < 1 || D < 1) return K3MOE_ERR_INVALID_ARG;
    if (D % 8) return K3MOE_ERR_SHAPE;
    if (!aligned16(h) || !aligned16(gamma) || !aligned16(out)) return K3MOE_ERR_ALIGN;
    return cuda_status(launch_rmsnorm(h, T, D, gamma, eps, out, static_cast<cudaStream_t>(stream)));
}

k3moe_status k3moe_gemm_bf16(const uint16_t* x, const uint16_t* w, int32_t T, int32_t N,
                             int32_t K, void* out, int32_t out_fp32, void* stream) {
    if (!x || !w || !out || T < 1 || N < 1 || K < 1) return K3MOE_ERR_INVALID_ARG;
    if (N % 128 || K % 64) return K3MOE_ERR_SHAPE;
    if (!aligned16(x) || !aligned16(w) || !aligned16(out)) return K3MOE_ERR_ALIGN;
    const cudaError_t e = launch_gemm_bf16(x, w, T, N, K, out, out_fp32 ? 1 : 0, nullptr,
                                           device_sms(), static_cast<cudaStream_t>(stream));
    if (e == cudaErrorNotSupported) return K3MOE_ERR_UNSUPPORTED;
    return cuda_status(e);
}

size_t k3moe_workspace_size(const k3moe_layer_desc* desc, int32_t T_max) {
    if (!desc || T_max < 1 || desc->E < 1 || desc->k < 1) return 0;
    return fwd_plan(desc, T_max).total;
}

size_t k3moe_host_staging_size(const k3moe_layer_desc* desc, int32_t T) {
    if (!desc || T < 1) return 0;
    const size_t width = desc->D > 0 ? desc->D : desc->d;
    return 2 * align_up(static_cast<size_t>(T) * width * 2);
}

namespace {

// The cached forward's view of the expert weights: the slot arrays, the
// expert -> slot map, and the device addresses of the host-resident arrays.
struct CachePlan {
    const k3moe_expert_cache* c = nullptr;
    CacheFillArgs fill{};
};

k3moe_status check_cache(const k3moe_layer_desc* d, const k3moe_expert_cache* c, int T, CachePlan* cp) {
    if (!c || c->reserved != 0 || !c->state) return K3MOE_ERR_INVALID_ARG;
    const long long need = std::min<long long>(d->E, static_cast<long long>(T) * d->k);
    if (c->slots < 1 || c->slots > d->E || c->slots < need) return K3MOE_ERR_SHAPE;
    // the slots hold the scales in the layout the kernels read: the caller's
    // prepared atoms or the canonical rows (not a per-call preparation)
    const ScaleSource ss = scale_source(d);
    if (ss == SCALES_CANON_PREP) return K3MOE_ERR_UNSUPPORTED;
    uint8_t* dst[6] = {c->w1_q, c->w3_q, c->w2_q, c->w1_s, c->w3_s, c->w2_s};
    for (uint8_t* q : dst) {
        if (!q) return K3MOE_ERR_INVALID_ARG;
        if (!aligned16(q)) return K3MOE_ERR_ALIGN;
    }
    if (!aligned32(c->w1_q) || !aligned32(c->w3_q) || !aligned32(c->w2_q) || !aligned16(c->state))
        return K3MOE_ERR_ALIGN;
    // the expert arrays of the layer are host memory, page-locked and mapped
    const bool prep = ss == SCALES_PREPARED;
    const void* src[6] = {d->w1_q, d->w3_q, d->w2_q, prep ? d->w1_sf : d->w1_s, prep ? d->w3_sf : d->w3_s,
                          prep ? d->w2_sf : d->w2_s};
    const uint8_t* dev[6];
    for (int i = 0; i < 6; ++i) {
        cudaPointerAttributes at{};
        if (cudaPointerGetAttributes(&at, src[i]) != cudaSuccess || at.type != cudaMemoryTypeHost ||
            !at.devicePointer || !at.hostPointer) {
            cudaGetLastError();
            return K3MOE_ERR_INVALID_ARG;
        }
        // the device address of the host byte src[i] (the allocation may start before it)
        const uint8_t* p = static_cast<const uint8_t*>(at.devicePointer) +
                           (static_cast<const uint8_t*>(src[i]) - static_cast<const uint8_t*>(at.hostPointer));
        if (!aligned16(p)) return K3MOE_ERR_ALIGN;
        dev[i] = p;
    }
    cp->c = c;
    for (int i = 0; i < 3; ++i) {
        cp->fill.src_q[i] = dev[i];
        cp->fill.src_sf[i] = dev[3 + i];
        cp->fill.dst_q[i] = dst[i];
        cp->fill.dst_sf[i] = dst[3 + i];
    }
    cp->fill.q_bytes = static_cast<size_t>(d->f) * (d->d / 2);
    // per expert, the same for all three matrices (w2 is [d, f], w1 and w3 [f, d])
    cp->fill.sf_bytes = prep ? prepared_sf_bytes(1, d->f, d->d) : static_cast<size_t>(d->f) * (d->d / 32);
    return K3MOE_OK;
}

// The forward; with idx_in / wts_in (device [T, k]) the caller's selection
// replaces the router (latent mode only).
k3moe_status forward_impl(const k3moe_layer_desc* desc, const k3moe_expert_cache* cache,
                          const uint16_t* hidden, int32_t T, uint16_t* out, void* ws, size_t ws_bytes,
                          void* stream, const int32_t* idx_in = nullptr, const float* wts_in = nullptr) {
    k3moe_status st = check_desc(desc);
    if (st != K3MOE_OK) return st;
    if (!hidden || !out || !ws || T < 1) return K3MOE_ERR_INVALID_ARG;
    if (!aligned16(hidden) || !aligned16(out) || !aligned16(ws)) return K3MOE_ERR_ALIGN;
    const bool routed = idx_in != nullptr;
    if (routed) {
        if (!wts_in) return K3MOE_ERR_INVALID_ARG;
        if (desc->D > 0) return K3MOE_ERR_UNSUPPORTED;
        if (!aligned16(idx_in) || !aligned16(wts_in)) return K3MOE_ERR_ALIGN;
    }
    const FwdPlan p = fwd_plan(desc, T);
    if (ws_bytes < p.total) return K3MOE_ERR_WORKSPACE;
    int path = desc->path;
    if (path == K3MOE_PATH_AUTO) path = T <= kStreamMaxT ? K3MOE_PATH_BLOCK_SCALED : K3MOE_PATH_BF16_DEQUANT;
    if (path == K3MOE_PATH_BLOCK_SCALED && T > kStreamMaxT) return K3MOE_ERR_UNSUPPORTED;
    // ggml blocks: the streaming kernels only, without a cache
    if (desc->format == K3MOE_FORMAT_GGML && (path != K3MOE_PATH_BLOCK_SCALED || cache)) return K3MOE_ERR_UNSUPPORTED;
    CachePlan cp;
    if (cache) {
        // the cache serves the streaming kernels only (few experts per call)
        if (path != K3MOE_PATH_BLOCK_SCALED) return K3MOE_ERR_UNSUPPORTED;
        if ((st = check_cache(desc, cache, T, &cp)) != K3MOE_OK) return st;
    }

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char* base = static_cast<char*>(ws);
    WsHeader* hdr = reinterpret_cast<WsHeader*>(base);
    const int sms = device_sms();
    std::lock_guard<std::mutex> trace_lock(g_trace.mu);
    trace_begin(s, reinterpret_cast<uint64_t*>(base + p.stamps));
    struct TraceEnd { ~TraceEnd() { trace_end(); } } trace_end_guard;
    auto at = [&](size_t off) { return static_cast<void*>(base + off); };
    cudaError_t e = cudaSuccess;
    const int inject = g_inject;  // armed for this forward only
    g_inject = 0;
    const ScaleSource ss = desc->format == K3MOE_FORMAT_GGML ? SCALES_PREPARED : scale_source(desc);
    if (ss == SCALES_CANON_PREP) {
        // widths that are not whole 512-input stages: the canonical rows are
        // rewritten as prepared atoms first (1/32 of the expert bytes)
        if ((e = launch_prepare_sf(desc->w1_s, desc->E, desc->f, desc->d, static_cast<uint8_t*>(at(p.sf1)), 0, s)) ||
            (e = launch_prepare_sf(desc->w3_s, desc->E, desc->f, desc->d, static_cast<uint8_t*>(at(p.sf3)), 0, s)) ||
            (e = launch_prepare_sf(desc->w2_s, desc->E, desc->d, desc->f, static_cast<uint8_t*>(at(p.sf2)), 0, s)))
            return cuda_status(e);
    }

    const uint16_t* x_router = hidden;
    const uint16_t* x_expert = hidden;
    uint16_t* latent_out = out;
    if (desc->D > 0) {
        uint16_t* hn = static_cast<uint16_t*>(at(p.hn));
        uint16_t* z = static_cast<uint16_t*>(at(p.z));
        if ((e = launch_rmsnorm(hidden, T, desc->D, desc->norm_gamma, desc->eps, hn, s))) return K3MOE_ERR_CUDA;
        e = launch_gemm_bf16(hn, desc->w_down, T, desc->d, desc->D, z, 0, hdr, sms, s, "latent_down");
        if (e == cudaErrorNotSupported) return K3MOE_ERR_UNSUPPORTED;
        if (e) return K3MOE_ERR_CUDA;
        x_router = hn;
        x_expert = z;
        latent_out = static_cast<uint16_t*>(at(p.m));
    }

    RouteArgs r{};
    r.x = x_router; r.T = T; r.d_r = desc->d_router; r.w = desc->router_w; r.bias = desc->router_b;
    r.E = desc->E; r.k = desc->k;
    r.idx = static_cast<int32_t*>(at(p.idx));
    r.wts = static_cast<float*>(at(p.wts));
    r.logits = static_cast<float*>(at(p.logits));
    r.hdr = hdr;
    int32_t* counts = static_cast<int32_t*>(at(p.counts));
    int32_t* offsets = static_cast<int32_t*>(at(p.offsets));
    int32_t* perm = static_cast<int32_t*>(at(p.perm));
    int32_t* inv = static_cast<int32_t*>(at(p.inv));
    int32_t* active = static_cast<int32_t*>(at(p.active));
    const bool fuse_prep = !routed && T <= kDecodeMaxT && path == K3MOE_PATH_BLOCK_SCALED && desc->D == 0;
    if (routed) {
        // the caller's selection: checked on the device by the histogram kernel
        // (an expert outside [0, E) records INVALID_ARG and becomes expert 0)
        // and permuted (the permutation also lists the active experts)
        const size_t P = static_cast<size_t>(T) * desc->k;
        if (cudaMemcpyAsync(r.idx, idx_in, P * 4, cudaMemcpyDeviceToDevice, s) ||
            cudaMemcpyAsync(r.wts, wts_in, P * 4, cudaMemcpyDeviceToDevice, s))
            return K3MOE_ERR_CUDA;
        if ((e = launch_permute(r.idx, T, desc->k, desc->E, counts, offsets, perm, inv, active, at(p.chunk), hdr, s,
                                1)))
            return K3MOE_ERR_CUDA;
    } else if (T <= kDecodeMaxT) {
        // decode needs only the active experts (listed by the top-k kernel); the
        // grouped path takes the full permutation
        r.active = path == K3MOE_PATH_BLOCK_SCALED ? active : nullptr;
        if (fuse_prep)
            mx_decode_xq_slots(at(p.dec), T, desc->E, desc->k, desc->d, desc->f, &r.xq, &r.xsf, &r.xq_n);
        if ((e = launch_route_small(r, s))) return cuda_status(e);
        if (path != K3MOE_PATH_BLOCK_SCALED &&
            (e = launch_permute(r.idx, T, desc->k, desc->E, counts, offsets, perm, inv, active, at(p.chunk), hdr, s)))
            return K3MOE_ERR_CUDA;
    } else {
        if (T >= 64 && desc->E % 128 == 0) {
            e = launch_gemm_bf16(x_router, desc->router_w, T, desc->E, desc->d_router, r.logits, 1,
                                 hdr, sms, s, "router_logits");
            if (e == cudaErrorNotSupported) e = launch_logits_simt(r, s);
        } else {
            e = launch_logits_simt(r, s);
        }
        if (e) return K3MOE_ERR_CUDA;
        if ((e = launch_topk(r, s))) return K3MOE_ERR_CUDA;
        if ((e = launch_permute(r.idx, T, desc->k, desc->E, counts, offsets, perm, inv, active,
                                at(p.chunk), hdr, s)))
            return K3MOE_ERR_CUDA;
    }

    // the weights the expert kernels read: the layer's arrays, or the cache's
    // slots after the missing experts were fetched into them
    const uint8_t *w1_q = desc->w1_q, *w3_q = desc->w3_q, *w2_q = desc->w2_q;
    const uint8_t *w1_sf = desc->w1_sf, *w3_sf = desc->w3_sf, *w2_sf = desc->w2_sf;
    int sf_canon = 0;
    if (ss == SCALES_CANON) {
        w1_sf = desc->w1_s; w3_sf = desc->w3_s; w2_sf = desc->w2_s;
        sf_canon = 1;
    } else if (ss == SCALES_CANON_PREP) {
        w1_sf = static_cast<const uint8_t*>(at(p.sf1));
        w3_sf = static_cast<const uint8_t*>(at(p.sf3));
        w2_sf = static_cast<const uint8_t*>(at(p.sf2));
    }
    const int32_t* slot_of = nullptr;
    int nslots = desc->E;
    if (cp.c) {
        if ((e = launch_cache_update(cp.c->state, desc->E, cp.c->slots, active, cp.fill, hdr, sms, s)))
            return cuda_status(e);
        w1_q = cp.c->w1_q; w3_q = cp.c->w3_q; w2_q = cp.c->w2_q;
        w1_sf = cp.c->w1_s; w3_sf = cp.c->w3_s; w2_sf = cp.c->w2_s;
        slot_of = cache_view(cp.c->state, desc->E, cp.c->slots).slot_of;
        nslots = cp.c->slots;
    }

    if (path == K3MOE_PATH_BLOCK_SCALED && T > kDecodeMaxT) {
        MxUnitsArgs a{};
        a.w1_q = w1_q; a.w3_q = w3_q; a.w2_q = w2_q;
        a.w1_sf = w1_sf; a.w3_sf = w3_sf; a.w2_sf = w2_sf; a.sf_canon = sf_canon;
        a.slot_of = slot_of; a.nslots = nslots;
        a.ggml = desc->format == K3MOE_FORMAT_GGML ? 1 : 0;
        a.x = x_expert; a.T = T; a.E = desc->E; a.k = desc->k; a.d = desc->d; a.f = desc->f;
        a.counts = counts; a.offsets = offsets; a.perm = perm; a.inv = inv; a.idx = r.idx; a.wts = r.wts;
        a.scratch = at(p.units);
        a.out = latent_out; a.hdr = hdr; a.num_sms = sms; a.inject = inject;
        e = launch_mx_units(a, s);
        if (e == cudaErrorNotSupported) return K3MOE_ERR_UNSUPPORTED;
        if (e) return cuda_status(e);
    } else if (path == K3MOE_PATH_BLOCK_SCALED) {
        MxDecodeArgs a{};
        a.w1_q = w1_q; a.w3_q = w3_q; a.w2_q = w2_q;
        a.w1_sf = w1_sf; a.w3_sf = w3_sf; a.w2_sf = w2_sf; a.sf_canon = sf_canon;
        a.slot_of = slot_of; a.nslots = nslots;
        a.ggml = desc->format == K3MOE_FORMAT_GGML ? 1 : 0;
        a.x = x_expert; a.xq_ready = fuse_prep ? 1 : 0;
        a.T = T; a.E = desc->E; a.k = desc->k; a.d = desc->d; a.f = desc->f;
        a.active = active; a.idx = r.idx; a.wts = r.wts;
        a.scratch = at(p.dec);
        a.out = latent_out; a.hdr = hdr; a.num_sms = sms; a.inject = inject;
        e = launch_mx_decode(a, s);
        if (e == cudaErrorNotSupported) return K3MOE_ERR_UNSUPPORTED;
        if (e) return cuda_status(e);
    } else {
        GroupedArgs g{};
        g.w1_q = desc->w1_q; g.w3_q = desc->w3_q; g.w2_q = desc->w2_q;
        g.w1_sf = w1_sf; g.w3_sf = w3_sf; g.w2_sf = w2_sf; g.sf_canon = sf_canon;
        g.x = x_expert; g.T = T; g.E = desc->E; g.k = desc->k; g.d = desc->d; g.f = desc->f;
        g.counts = counts; g.offsets = offsets; g.perm = perm; g.inv = inv; g.wts = r.wts;
        g.xp = static_cast<uint16_t*>(at(p.xp));
        g.xp_exp = static_cast<int32_t*>(at(p.xp_exp));
        g.hf = static_cast<float*>(at(p.hb));
        g.h_amax = static_cast<uint32_t*>(at(p.h_amax));
        g.hp = static_cast<uint16_t*>(at(p.hp));
        g.hp_exp = static_cast<int32_t*>(at(p.hp_exp));
        g.y = static_cast<float*>(at(p.y));
        g.tiles = static_cast<int32_t*>(at(p.tiles));
        g.tiles_cap = p.tiles_cap;
        g.out = latent_out; g.hdr = hdr; g.num_sms = sms;
        e = launch_grouped(g, s);
        if (e == cudaErrorNotSupported) return K3MOE_ERR_UNSUPPORTED;
        if (e) return K3MOE_ERR_CUDA;
    }

    if (desc->D > 0) {
        e = launch_gemm_bf16(latent_out, desc->w_up, T, desc->D, desc->d, out, 0, hdr, sms, s, "latent_up");
        if (e == cudaErrorNotSupported) return K3MOE_ERR_UNSUPPORTED;
        if (e) return K3MOE_ERR_CUDA;
    }
    return K3MOE_OK;
}

}  // namespace

k3moe_status k3moe_forward(const k3moe_layer_desc* desc, const uint16_t* hidden, int32_t T,
                           uint16_t* out, void* ws, size_t ws_bytes, void* stream) {
    return forward_impl(desc, nullptr, hidden, T, out, ws, ws_bytes, stream);
}

k3moe_status k3moe_forward_routed(const k3moe_layer_desc* desc, const uint16_t* hidden, int32_t T,
                                  const int32_t* idx, const float* wts, uint16_t* out, void* ws, size_t ws_bytes,
                                  void* stream) {
    if (!idx || !wts) return K3MOE_ERR_INVALID_ARG;
    return forward_impl(desc, nullptr, hidden, T, out, ws, ws_bytes, stream, idx, wts);
}

size_t k3moe_cache_state_size(int32_t E, int32_t slots) {
    if (E < 1 || slots < 1) return 0;
    return cache_state_bytes(E, slots);
}

k3moe_status k3moe_cache_init(void* state, int32_t E, int32_t slots, void* stream) {
    if (!state || E < 1 || slots < 1) return K3MOE_ERR_INVALID_ARG;
    if (slots > E || E > 1024) return K3MOE_ERR_SHAPE;
    if (!aligned16(state)) return K3MOE_ERR_ALIGN;
    return cuda_status(launch_cache_init(state, E, slots, static_cast<cudaStream_t>(stream)));
}

k3moe_status k3moe_forward_cached(const k3moe_layer_desc* desc, const k3moe_expert_cache* cache,
                                  const uint16_t* hidden, int32_t T, uint16_t* out, void* ws,
                                  size_t ws_bytes, void* stream) {
    if (!cache) return K3MOE_ERR_INVALID_ARG;
    return forward_impl(desc, cache, hidden, T, out, ws, ws_bytes, stream);
}

k3moe_status k3moe_cache_read_stats(const void* state, void* stream, k3moe_cache_stats* out) {
    if (!state || !out) return K3MOE_ERR_INVALID_ARG;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return K3MOE_ERR_CUDA;
    CacheHeader h;
    if (cudaMemcpy(&h, state, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return K3MOE_ERR_CUDA;
    if (h.magic != kCacheMagic) return K3MOE_ERR_INVALID_ARG;
    out->calls = h.calls;
    out->hits = h.hits;
    out->misses = h.misses;
    out->bytes = h.bytes;
    out->last_hits = h.last_hit;
    out->last_misses = h.last_miss;
    return K3MOE_OK;
}

namespace {
// k3moe_forward_host replays a cached CUDA graph of the forward when a call
// repeats the last ones' arguments: its staging buffers sit at fixed offsets
// of the workspace, so the same descriptor contents, workspace, token count,
// stream and device mean the same kernels on the same addresses.  A graph
// references the buffers, not their contents, so new weights written in
// place are read by the next replay.  At most kHostGraphs entries, the least
// recently used one replaced.  For small batches (kHostStageMax bytes of
// tokens or less) the entry also owns two page-locked host buffers and the
// graph copies the tokens in from one and the output out to the other, so a
// call is two host memcpys, one graph launch and one wait instead of three
// stream operations; larger batches copy straight from and to the caller's
// buffers around the graph.  An entry in use by a call (it may run in another
// host thread) is never replaced: a new graph that finds every entry in use
// is not kept.
constexpr size_t kHostStageMax = 1 << 20;
struct HostGraph {
    k3moe_layer_desc desc;
    const void* ws;
    size_t ws_bytes;
    int32_t T;
    cudaStream_t s;
    int dev;
    cudaGraphExec_t exec;
    void* pin_in;  // page-locked staging of a small batch, or null
    void* pin_out;
    uint64_t used;
    int busy;      // calls using the entry now
};
struct HostGraphHit {
    cudaGraphExec_t exec;
    void* pin_in;
    void* pin_out;
    int index;     // the entry, held until host_graph_release (-1: none)
};
constexpr int kHostGraphs = 8;
std::mutex g_host_mu;
HostGraph g_host[kHostGraphs] = {};
uint64_t g_host_clock = 0;

bool same_key(const HostGraph& h, const k3moe_layer_desc* d, const void* ws, size_t ws_bytes, int32_t T,
              cudaStream_t s, int dev) {
    return h.exec && h.ws == ws && h.ws_bytes == ws_bytes && h.T == T && h.s == s && h.dev == dev &&
           std::memcmp(&h.desc, d, sizeof(k3moe_layer_desc)) == 0;
}

// the cached graph for these arguments (exec null when there is none), held
// for the caller until host_graph_release
HostGraphHit host_graph_find(const k3moe_layer_desc* d, const void* ws, size_t ws_bytes, int32_t T,
                             cudaStream_t s, int dev) {
    std::lock_guard<std::mutex> lock(g_host_mu);
    for (int i = 0; i < kHostGraphs; ++i) {
        HostGraph& h = g_host[i];
        if (same_key(h, d, ws, ws_bytes, T, s, dev)) {
            h.used = ++g_host_clock;
            ++h.busy;
            return {h.exec, h.pin_in, h.pin_out, i};
        }
    }
    return {nullptr, nullptr, nullptr, -1};
}

void host_graph_release(int index) {
    if (index < 0) return;
    std::lock_guard<std::mutex> lock(g_host_mu);
    --g_host[index].busy;
}

// releases a found entry when the call returns
struct HostGraphHold {
    int index;
    ~HostGraphHold() { host_graph_release(index); }
};

// Copies n 16-bit words between device memory and mapped page-locked host
// memory: for a batch of a few KiB the loads and stores of one small grid
// reach the host over the chip-to-chip link sooner than a copy-engine
// transfer is set up.  16-byte words when both ends allow, else 2-byte ones.
__global__ void stage_copy_kernel(const uint16_t* __restrict__ src, uint16_t* __restrict__ dst, size_t n) {
    const size_t tid = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
    if (((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 15) == 0) {
        const size_t n16 = n / 8;
        const uint4* s16 = reinterpret_cast<const uint4*>(src);
        uint4* d16 = reinterpret_cast<uint4*>(dst);
        for (size_t i = tid; i < n16; i += stride) d16[i] = s16[i];
        for (size_t i = n16 * 8 + tid; i < n; i += stride) dst[i] = src[i];
    } else {
        for (size_t i = tid; i < n; i += stride) dst[i] = src[i];
    }
}

cudaError_t stage_copy(const void* src, void* dst, size_t bytes, cudaStream_t s) {
    const size_t n = bytes / 2;
    const int threads = 256;
    const size_t want = (n / 8 + threads - 1) / threads;
    const int blocks = static_cast<int>(want < 1 ? 1 : (want > 256 ? 256 : want));
    stage_copy_kernel<<<blocks, threads, 0, s>>>(static_cast<const uint16_t*>(src), static_cast<uint16_t*>(dst), n);
    return cudaGetLastError();
}

void free_pinned(void* a, void* b) {
    if (a) cudaFreeHost(a);
    if (b) cudaFreeHost(b);
}

// capture the forward (nothing runs) on a private stream and keep the graph;
// with staging buffers the copies from and to them are part of the graph
void host_graph_add(const k3moe_layer_desc* d, uint16_t* in_dev, int32_t T, uint16_t* out_dev, void* ws,
                    size_t need, size_t ws_bytes, size_t bytes, cudaStream_t s, int dev) {
    void* pin_in = nullptr;
    void* pin_out = nullptr;
    void* map_in = nullptr;  // their device addresses
    void* map_out = nullptr;
    if (bytes <= kHostStageMax && (cudaHostAlloc(&pin_in, bytes, cudaHostAllocMapped) != cudaSuccess ||
                                   cudaHostAlloc(&pin_out, bytes, cudaHostAllocMapped) != cudaSuccess ||
                                   cudaHostGetDevicePointer(&map_in, pin_in, 0) != cudaSuccess ||
                                   cudaHostGetDevicePointer(&map_out, pin_out, 0) != cudaSuccess)) {
        // no staging: the graph holds the forward alone
        free_pinned(pin_in, pin_out);
        pin_in = pin_out = nullptr;
        cudaGetLastError();
    }
    cudaStream_t cs = nullptr;
    if (cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking) != cudaSuccess) {
        cudaGetLastError();
        free_pinned(pin_in, pin_out);
        return;
    }
    cudaGraph_t g = nullptr;
    cudaGraphExec_t exec = nullptr;
    bool ok = cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal) == cudaSuccess;
    if (ok) {
        if (pin_in) ok = stage_copy(map_in, in_dev, bytes, cs) == cudaSuccess;
        ok = ok && k3moe_forward(d, in_dev, T, out_dev, ws, need, cs) == K3MOE_OK;
        if (pin_out) ok = ok && stage_copy(out_dev, map_out, bytes, cs) == cudaSuccess;
        ok = cudaStreamEndCapture(cs, &g) == cudaSuccess && ok;
    }
    ok = ok && cudaGraphInstantiate(&exec, g, 0) == cudaSuccess;
    if (g) cudaGraphDestroy(g);
    cudaStreamDestroy(cs);
    if (!ok) {
        if (exec) cudaGraphExecDestroy(exec);
        free_pinned(pin_in, pin_out);
        cudaGetLastError();
        return;
    }
    std::lock_guard<std::mutex> lock(g_host_mu);
    HostGraph* slot = nullptr;  // an empty entry, else the least recently used one not in use
    for (auto& h : g_host) {
        if (h.busy > 0) continue;
        if (!slot || !h.exec || (slot->exec && h.used < slot->used)) slot = &h;
    }
    if (!slot) {
        cudaGraphExecDestroy(exec);
        free_pinned(pin_in, pin_out);
        return;
    }
    if (slot->exec) cudaGraphExecDestroy(slot->exec);
    free_pinned(slot->pin_in, slot->pin_out);
    slot->desc = *d;
    slot->ws = ws;
    slot->ws_bytes = ws_bytes;
    slot->T = T;
    slot->s = s;
    slot->dev = dev;
    slot->exec = exec;
    slot->pin_in = pin_in;
    slot->pin_out = pin_out;
    slot->used = ++g_host_clock;
    slot->busy = 0;
}
}  // namespace

k3moe_status k3moe_forward_host(const k3moe_layer_desc* desc, const uint16_t* hidden_host,
                                int32_t T, uint16_t* out_host, void* ws, size_t ws_bytes,
                                void* stream) {
    k3moe_status st = check_desc(desc);
    if (st != K3MOE_OK) return st;
    if (!hidden_host || !out_host || !ws || T < 1) return K3MOE_ERR_INVALID_ARG;
    const size_t need = k3moe_workspace_size(desc, T);
    const size_t stage = k3moe_host_staging_size(desc, T);
    if (ws_bytes < need + stage) return K3MOE_ERR_WORKSPACE;
    const size_t width = desc->D > 0 ? desc->D : desc->d;
    const size_t bytes = static_cast<size_t>(T) * width * 2;
    char* base = static_cast<char*>(ws);
    uint16_t* in_dev = reinterpret_cast<uint16_t*>(base + need);
    uint16_t* out_dev = reinterpret_cast<uint16_t*>(base + need + stage / 2);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return K3MOE_ERR_CUDA;
    // a graph only when nothing else would record this forward: no tracing and
    // no capture of the caller's stream
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    const bool plain = g_trace.mode == 0 && g_inject == 0 && cudaStreamIsCapturing(s, &cap) == cudaSuccess &&
                       cap == cudaStreamCaptureStatusNone;
    const HostGraphHit hit =
        plain ? host_graph_find(desc, ws, ws_bytes, T, s, dev) : HostGraphHit{nullptr, nullptr, nullptr, -1};
    const HostGraphHold hold{hit.index};
    if (hit.exec && hit.pin_in) {
        // the graph copies in from and out to its own page-locked buffers
        std::memcpy(hit.pin_in, hidden_host, bytes);
        if (cudaGraphLaunch(hit.exec, s) != cudaSuccess) return K3MOE_ERR_CUDA;
        const k3moe_status done = cuda_status(cudaStreamSynchronize(s));
        if (done == K3MOE_OK) std::memcpy(out_host, hit.pin_out, bytes);
        return done;
    }
    if (cudaMemcpyAsync(in_dev, hidden_host, bytes, cudaMemcpyHostToDevice, s)) return K3MOE_ERR_CUDA;
    if (hit.exec) {
        if (cudaGraphLaunch(hit.exec, s) != cudaSuccess) return K3MOE_ERR_CUDA;
    } else {
        st = k3moe_forward(desc, in_dev, T, out_dev, ws, need, stream);
        if (st != K3MOE_OK) return st;
        if (plain) host_graph_add(desc, in_dev, T, out_dev, ws, need, ws_bytes, bytes, s, dev);
    }
    if (cudaMemcpyAsync(out_host, out_dev, bytes, cudaMemcpyDeviceToHost, s)) return K3MOE_ERR_CUDA;
    return cuda_status(cudaStreamSynchronize(s));
}

namespace {
struct ForwardGraph {
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
};
}  // namespace

namespace {
k3moe_status graph_create(const k3moe_layer_desc* desc, const k3moe_expert_cache* cache,
                          const uint16_t* hidden, int32_t T, uint16_t* out, void* ws, size_t ws_bytes,
                          void** graph_out) {
    if (!graph_out) return K3MOE_ERR_INVALID_ARG;
    *graph_out = nullptr;
    // the set-up forward runs on a private stream: work the caller queued on
    // its own streams (which may use the same workspace or cache) finishes first
    if (cudaDeviceSynchronize() != cudaSuccess) return K3MOE_ERR_CUDA;
    cudaStream_t cs = nullptr;
    if (cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking) != cudaSuccess) return K3MOE_ERR_CUDA;
    // one uncaptured forward: argument checks and one-time set-up
    k3moe_status st = forward_impl(desc, cache, hidden, T, out, ws, ws_bytes, cs);
    if (st == K3MOE_OK && cudaStreamSynchronize(cs) != cudaSuccess) st = K3MOE_ERR_CUDA;
    ForwardGraph* fg = nullptr;
    if (st == K3MOE_OK) {
        fg = new ForwardGraph();
        if (cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
            st = K3MOE_ERR_CUDA;
        } else {
            st = forward_impl(desc, cache, hidden, T, out, ws, ws_bytes, cs);
            const cudaError_t e = cudaStreamEndCapture(cs, &fg->graph);
            if (st == K3MOE_OK && e != cudaSuccess) st = K3MOE_ERR_CUDA;
        }
        if (st == K3MOE_OK && cudaGraphInstantiate(&fg->exec, fg->graph, 0) != cudaSuccess)
            st = K3MOE_ERR_CUDA;
    }
    cudaStreamDestroy(cs);
    if (st != K3MOE_OK) {
        if (fg) {
            if (fg->exec) cudaGraphExecDestroy(fg->exec);
            if (fg->graph) cudaGraphDestroy(fg->graph);
            delete fg;
        }
        cudaGetLastError();  // leave no pending error behind
        return st;
    }
    *graph_out = fg;
    return K3MOE_OK;
}
}  // namespace

k3moe_status k3moe_graph_create(const k3moe_layer_desc* desc, const uint16_t* hidden, int32_t T,
                                uint16_t* out, void* ws, size_t ws_bytes, void** graph_out) {
    return graph_create(desc, nullptr, hidden, T, out, ws, ws_bytes, graph_out);
}

k3moe_status k3moe_graph_create_cached(const k3moe_layer_desc* desc, const k3moe_expert_cache* cache,
                                       const uint16_t* hidden, int32_t T, uint16_t* out, void* ws,
                                       size_t ws_bytes, void** graph_out) {
    if (!cache) return K3MOE_ERR_INVALID_ARG;
    return graph_create(desc, cache, hidden, T, out, ws, ws_bytes, graph_out);
}

k3moe_status k3moe_graph_launch(void* graph, void* stream) {
    if (!graph) return K3MOE_ERR_INVALID_ARG;
    return cuda_status(cudaGraphLaunch(static_cast<ForwardGraph*>(graph)->exec,
                                       static_cast<cudaStream_t>(stream)));
}

k3moe_status k3moe_graph_destroy(void* graph) {
    if (!graph) return K3MOE_ERR_INVALID_ARG;
    ForwardGraph* fg = static_cast<ForwardGraph*>(graph);
    cudaError_t e1 = cudaGraphExecDestroy(fg->exec);
    cudaError_t e2 = cudaGraphDestroy(fg->graph);
    delete fg;
    return (e1 == cudaSuccess && e2 == cudaSuccess) ? K3MOE_OK : K3MOE_ERR_CUDA;
}

k3moe_status k3moe_forward_routing(const k3moe_layer_desc* desc, const void* ws, int32_t T,
                                   int32_t* idx_out, float* w_out, float* logits_out,
                                   void* stream) {
    if (!desc || !ws || !idx_out || !w_out || T < 1 || desc->E < 1 || desc->k < 1)
        return K3MOE_ERR_INVALID_ARG;
    const FwdPlan p = fwd_plan(desc, T);
    const char* base = static_cast<const char*>(ws);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t P = static_cast<size_t>(T) * desc->k;
    if (cudaMemcpyAsync(idx_out, base + p.idx, P * 4, cudaMemcpyDeviceToDevice, s)) return K3MOE_ERR_CUDA;
    if (cudaMemcpyAsync(w_out, base + p.wts, P * 4, cudaMemcpyDeviceToDevice, s)) return K3MOE_ERR_CUDA;
    if (logits_out &&
        cudaMemcpyAsync(logits_out, base + p.logits, static_cast<size_t>(T) * desc->E * 4,
                        cudaMemcpyDeviceToDevice, s))
        return K3MOE_ERR_CUDA;
    return K3MOE_OK;
}

k3moe_status k3moe_forward_intermediates(const k3moe_layer_desc* desc, const void* ws, int32_t T,
                                         uint16_t* hn_out, uint16_t* z_out, uint16_t* m_out, void* stream) {
    if (!desc || !ws || T < 1 || desc->E < 1 || desc->k < 1) return K3MOE_ERR_INVALID_ARG;
    if (desc->D <= 0) return K3MOE_ERR_UNSUPPORTED;  // latent mode keeps no intermediates
    const FwdPlan p = fwd_plan(desc, T);
    const char* base = static_cast<const char*>(ws);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t nD = static_cast<size_t>(T) * desc->D * 2, nd = static_cast<size_t>(T) * desc->d * 2;
    if (hn_out && cudaMemcpyAsync(hn_out, base + p.hn, nD, cudaMemcpyDeviceToDevice, s)) return K3MOE_ERR_CUDA;
    if (z_out && cudaMemcpyAsync(z_out, base + p.z, nd, cudaMemcpyDeviceToDevice, s)) return K3MOE_ERR_CUDA;
    if (m_out && cudaMemcpyAsync(m_out, base + p.m, nd, cudaMemcpyDeviceToDevice, s)) return K3MOE_ERR_CUDA;
    return K3MOE_OK;
}

k3moe_status k3moe_get_status(void* ws, void* stream, int32_t* device_status) {
    if (!ws || !device_status) return K3MOE_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return K3MOE_ERR_CUDA;
    int32_t st = 0;
    if (cudaMemcpy(&st, ws, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return K3MOE_ERR_CUDA;
    *device_status = st;
    if (st != 0 && cudaMemset(ws, 0, 8) != cudaSuccess) return K3MOE_ERR_CUDA;
    return K3MOE_OK;
}

}  // extern "C"
