// Host side of the spec_tree library: errors, tree encoding, device status,
// tracing, and the Philox inspection entry point.
#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "common.cuh"
#include "philox.cuh"

namespace spec {

// ---------------------------------------------------------------- errors

static thread_local std::string g_error;

void set_error(const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_error = buf;
}

void clear_error() { g_error.clear(); }

spec_status fail(spec_status st, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_error = buf;
    return st;
}

int device_sm_count() {
    static std::mutex mu;
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    std::lock_guard<std::mutex> lock(mu);
    if (cached[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        cached[dev] = n;
    }
    return cached[dev];
}

spec_status check_tree(const spec_tree* t) {
    if (!t) return fail(SPEC_EINVAL, "tree is NULL");
    if (t->T < 1 || t->T > SPEC_MAX_T) return fail(SPEC_EINVAL, "tree->T = %d out of 1..%d", t->T, SPEC_MAX_T);
    if (t->max_depth < 0 || t->max_depth > SPEC_MAX_DEPTH || t->words != (t->T + 63) / 64)
        return fail(SPEC_EINVAL, "tree header is inconsistent (was it filled by spec_tree_build?)");
    if (!t->parent || !t->depth || !t->rank || !t->anc || !t->internal || !t->internal_off || !t->row_of ||
        !t->child_off || !t->child_idx)
        return fail(SPEC_EINVAL, "tree has NULL device tables (was it filled by spec_tree_build?)");
    return SPEC_OK;
}

cudaError_t reset_device_status(void* ws, cudaStream_t s) { return cudaMemsetAsync(ws, 0, 16, s); }

// ---------------------------------------------------------------- tracing

struct TraceState {
    bool on = false;
    int capacity = 0;
    int used = 0;
    std::vector<cudaEvent_t> ev;     // 2 per launch
    std::vector<std::string> names;
};
static TraceState g_trace;
static std::atomic<int64_t> g_launches{0};

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

bool trace_active() { return g_trace.on; }

void trace_before(cudaStream_t s) {
    if (!g_trace.on || g_trace.used >= g_trace.capacity) return;
    cudaEventRecord(g_trace.ev[2 * g_trace.used], s);
}

void trace_after(cudaStream_t s, const char* name) {
    if (!g_trace.on || g_trace.used >= g_trace.capacity) return;
    cudaEventRecord(g_trace.ev[2 * g_trace.used + 1], s);
    g_trace.names[g_trace.used] = name;
    ++g_trace.used;
}

// ---------------------------------------------------------------- tree encoding

namespace {

struct TreeLayout {
    size_t parent, depth, rank, internal, internal_off, row_of, child_off, child_idx, anc, total;
};

TreeLayout tree_layout(int32_t T) {
    TreeLayout L{};
    const int words = (T + 63) / 64;
    size_t off = 0;
    auto take = [&](size_t bytes) { size_t at = off; off = round_up(off + bytes, 16); return at; };
    L.parent = take(sizeof(int32_t) * T);
    L.depth = take(sizeof(int32_t) * T);
    L.rank = take(sizeof(int32_t) * T);
    L.internal = take(sizeof(int32_t) * T);
    L.internal_off = take(sizeof(int32_t) * (SPEC_MAX_DEPTH + 2));
    L.row_of = take(sizeof(int32_t) * T);
    L.child_off = take(sizeof(int32_t) * (T + 1));
    L.child_idx = take(sizeof(int32_t) * std::max(T - 1, 1));
    L.anc = take(sizeof(uint64_t) * static_cast<size_t>(T) * words);
    L.total = off;
    return L;
}

}  // namespace
}  // namespace spec

using namespace spec;

extern "C" {

const char* spec_last_error(void) { return g_error.c_str(); }

size_t spec_tree_device_bytes(int32_t T) {
    if (T < 1 || T > SPEC_MAX_T) return 0;
    return tree_layout(T).total;
}

spec_status spec_tree_build(const int32_t* parent, const int32_t* rank, int32_t T, void* d_buf, size_t d_bytes,
                            spec_tree* out, spec_stream_t s_) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(s_);
    clear_error();
    if (!parent || !out) return fail(SPEC_EINVAL, "parent and out must not be NULL");
    if (T < 1 || T > SPEC_MAX_T) return fail(SPEC_EINVAL, "T = %d out of 1..%d", T, SPEC_MAX_T);
    if (!d_buf) return fail(SPEC_EINVAL, "d_buf is NULL");
    if (!aligned16(d_buf)) return fail(SPEC_EALIGN, "d_buf is not 16-byte aligned");
    const TreeLayout L = tree_layout(T);
    if (d_bytes < L.total) return fail(SPEC_EWORKSPACE, "d_bytes = %zu < %zu needed", d_bytes, L.total);

    // validate and derive on the host
    if (parent[0] != -1) return fail(SPEC_ETREE, "parent[0] = %d, must be -1", parent[0]);
    std::vector<int32_t> depth(T, 0), rk(T, 0), nkids(T, 0);
    for (int i = 1; i < T; ++i) {
        if (parent[i] < 0 || parent[i] >= i) return fail(SPEC_ETREE, "parent[%d] = %d not in [0, %d)", i, parent[i], i);
        depth[i] = depth[parent[i]] + 1;
        if (depth[i] > SPEC_MAX_DEPTH) return fail(SPEC_ETREE, "node %d is deeper than %d", i, SPEC_MAX_DEPTH);
        rk[i] = rank ? rank[i] : nkids[parent[i]];
        if (rk[i] < 0) return fail(SPEC_ETREE, "rank[%d] = %d is negative", i, rk[i]);
        ++nkids[parent[i]];
    }
    std::vector<int32_t> child_off(T + 1, 0);
    for (int u = 0; u < T; ++u) child_off[u + 1] = child_off[u] + nkids[u];
    std::vector<int32_t> child_idx(std::max(T - 1, 1), 0), fill(child_off.begin(), child_off.end() - 1);
    for (int i = 1; i < T; ++i) child_idx[fill[parent[i]]++] = i;
    for (int u = 0; u < T; ++u)
        for (int a = child_off[u]; a < child_off[u + 1]; ++a)
            for (int b = a + 1; b < child_off[u + 1]; ++b)
                if (rk[child_idx[a]] == rk[child_idx[b]])
                    return fail(SPEC_ETREE, "children %d and %d of node %d share rank %d", child_idx[a],
                                child_idx[b], u, rk[child_idx[a]]);

    spec_tree t{};
    t.T = T;
    t.words = (T + 63) / 64;
    t.max_depth = *std::max_element(depth.begin(), depth.end());
    for (int d = 0; d <= SPEC_MAX_DEPTH; ++d) t.max_rank_at_depth[d] = -1;
    std::vector<int32_t> internal, internal_off(SPEC_MAX_DEPTH + 2, 0), row_of(T, -1);
    for (int d = 0; d <= SPEC_MAX_DEPTH; ++d) {
        internal_off[d] = static_cast<int32_t>(internal.size());
        for (int u = 0; u < T; ++u) {
            if (depth[u] != d) continue;
            ++t.n_at_depth[d];
            if (d > 0) t.max_rank_at_depth[d] = std::max(t.max_rank_at_depth[d], rk[u]);
            if (nkids[u] > 0) {
                row_of[u] = t.n_internal_at_depth[d]++;
                internal.push_back(u);
            }
        }
    }
    internal_off[SPEC_MAX_DEPTH + 1] = static_cast<int32_t>(internal.size());
    t.n_internal = static_cast<int32_t>(internal.size());
    internal.resize(T, 0);

    std::vector<uint64_t> anc(static_cast<size_t>(T) * t.words, 0);
    for (int i = 0; i < T; ++i)
        for (int j = i; j != -1; j = (j == 0 ? -1 : parent[j])) anc[static_cast<size_t>(i) * t.words + j / 64] |= 1ull << (j % 64);

    std::vector<unsigned char> host(L.total, 0);
    auto put = [&](size_t off, const void* src, size_t bytes) { std::memcpy(host.data() + off, src, bytes); };
    std::vector<int32_t> par(parent, parent + T);
    put(L.parent, par.data(), sizeof(int32_t) * T);
    put(L.depth, depth.data(), sizeof(int32_t) * T);
    put(L.rank, rk.data(), sizeof(int32_t) * T);
    put(L.internal, internal.data(), sizeof(int32_t) * T);
    put(L.internal_off, internal_off.data(), sizeof(int32_t) * (SPEC_MAX_DEPTH + 2));
    put(L.row_of, row_of.data(), sizeof(int32_t) * T);
    put(L.child_off, child_off.data(), sizeof(int32_t) * (T + 1));
    put(L.child_idx, child_idx.data(), sizeof(int32_t) * child_idx.size());
    put(L.anc, anc.data(), sizeof(uint64_t) * anc.size());

    SPEC_CUDA_TRY(cudaMemcpyAsync(d_buf, host.data(), L.total, cudaMemcpyHostToDevice, s));
    SPEC_CUDA_TRY(cudaStreamSynchronize(s));

    unsigned char* base = static_cast<unsigned char*>(d_buf);
    t.parent = reinterpret_cast<const int32_t*>(base + L.parent);
    t.depth = reinterpret_cast<const int32_t*>(base + L.depth);
    t.rank = reinterpret_cast<const int32_t*>(base + L.rank);
    t.internal = reinterpret_cast<const int32_t*>(base + L.internal);
    t.internal_off = reinterpret_cast<const int32_t*>(base + L.internal_off);
    t.row_of = reinterpret_cast<const int32_t*>(base + L.row_of);
    t.child_off = reinterpret_cast<const int32_t*>(base + L.child_off);
    t.child_idx = reinterpret_cast<const int32_t*>(base + L.child_idx);
    t.anc = reinterpret_cast<const uint64_t*>(base + L.anc);
    *out = t;
    return SPEC_OK;
}

spec_status spec_read_device_status(const void* ws, int32_t* status, spec_stream_t s_) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(s_);
    clear_error();
    if (!ws || !status) return fail(SPEC_EINVAL, "ws and status must not be NULL");
    int32_t v = 0;
    SPEC_CUDA_TRY(cudaMemcpyAsync(&v, ws, sizeof(v), cudaMemcpyDeviceToHost, s));
    SPEC_CUDA_TRY(cudaStreamSynchronize(s));
    *status = v;
    return SPEC_OK;
}

spec_status spec_trace_begin(int32_t capacity) {
    clear_error();
    if (capacity < 1 || capacity > (1 << 20)) return fail(SPEC_EINVAL, "capacity %d out of 1..2^20", capacity);
    for (cudaEvent_t e : g_trace.ev) cudaEventDestroy(e);
    g_trace = TraceState{};
    g_trace.ev.resize(2 * static_cast<size_t>(capacity));
    g_trace.names.resize(capacity);
    for (auto& e : g_trace.ev) SPEC_CUDA_TRY(cudaEventCreate(&e));
    g_trace.capacity = capacity;
    g_trace.on = true;
    return SPEC_OK;
}

int32_t spec_trace_end(spec_trace_entry* out, int32_t max_entries) {
    clear_error();
    if (!g_trace.on) { fail(SPEC_EINVAL, "tracing is not on"); return -1; }
    g_trace.on = false;
    std::vector<spec_trace_entry> agg;
    for (int i = 0; i < g_trace.used; ++i) {
        if (cudaEventSynchronize(g_trace.ev[2 * i + 1]) != cudaSuccess) { fail(SPEC_ECUDA, "event sync failed"); return -1; }
        float ms = 0.f;
        cudaEventElapsedTime(&ms, g_trace.ev[2 * i], g_trace.ev[2 * i + 1]);
        auto it = std::find_if(agg.begin(), agg.end(),
                               [&](const spec_trace_entry& e) { return g_trace.names[i] == e.name; });
        if (it == agg.end()) {
            spec_trace_entry e{};
            std::snprintf(e.name, sizeof(e.name), "%s", g_trace.names[i].c_str());
            agg.push_back(e);
            it = agg.end() - 1;
        }
        it->launches += 1;
        it->total_ms += ms;
    }
    for (cudaEvent_t e : g_trace.ev) cudaEventDestroy(e);
    g_trace = TraceState{};
    const int n = std::min<int>(static_cast<int>(agg.size()), std::max(max_entries, 0));
    for (int i = 0; i < n && out; ++i) out[i] = agg[i];
    return static_cast<int32_t>(agg.size());
}

int64_t spec_launch_count(void) { return g_launches.load(); }

}  // extern "C"

// ---------------------------------------------------------------- Philox inspection

namespace spec {
__global__ void k_philox_uniform(uint64_t seed, uint64_t offset, int B, int T, float* u_accept, float* u_sample) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= B * T) return;
    const int b = i / T, c = i % T;
    const spec::Philox4 r = spec::spec_draw(seed, offset, static_cast<uint32_t>(c), static_cast<uint32_t>(b));
    u_accept[i] = spec::uniform24(r.w[0]);
    if (c == 0) u_sample[b] = spec::uniform24(r.w[1]);
}
}  // namespace spec

extern "C" spec_status spec_philox_uniform(uint64_t seed, uint64_t offset, int32_t B, int32_t T, float* u_accept,
                                           float* u_sample, spec_stream_t s_) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(s_);
    clear_error();
    if (B < 1 || T < 1 || static_cast<int64_t>(B) * T > (1ll << 30)) return fail(SPEC_EINVAL, "B = %d, T = %d out of range", B, T);
    if (!u_accept || !u_sample) return fail(SPEC_EINVAL, "outputs must not be NULL");
    if (!aligned4(u_accept) || !aligned4(u_sample)) return fail(SPEC_EALIGN, "outputs must be 4-byte aligned");
    const int n = B * T;
    SPEC_CUDA_TRY(launch("philox_uniform", k_philox_uniform, dim3((n + 255) / 256), dim3(256), 0, s, seed, offset, B, T,
                         u_accept, u_sample));
    return SPEC_OK;
}

// ---------------------------------------------------------------- bounded-wait self-test

#include "tc.cuh"

namespace spec {
// One thread waits on a shared-memory barrier that nothing completes; the
// bounded wait used by the tensor-core kernels gives up after limit_ns and
// records SPEC_ETIMEOUT in the workspace status word.
__global__ void k_selftest_timeout(void* ws, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x != 0) return;
    tc::mbar_init(&bar, 1);
    tc::fence_mbar_init();
    if (!tc::mbar_wait(&bar, 0, limit_ns)) flag_status(ws, SPEC_ETIMEOUT);
}
}  // namespace spec

extern "C" spec_status spec_selftest_timeout(void* ws, uint64_t limit_ns, spec_stream_t s_) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(s_);
    clear_error();
    if (!ws) return fail(SPEC_EINVAL, "ws must not be NULL");
    if (!aligned16(ws)) return fail(SPEC_EALIGN, "ws must be 16-byte aligned");
    if (limit_ns > 1000000000ull) limit_ns = 1000000000ull;
    SPEC_CUDA_TRY(reset_device_status(ws, s));
    SPEC_CUDA_TRY(launch("selftest_timeout", k_selftest_timeout, dim3(1), dim3(32), 0, s, ws, limit_ns));
    return SPEC_OK;
}
