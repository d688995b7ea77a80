// KV commit of the accepted path.
//
// Speculative Decoding (thegustafson.com), section "The acceptance criterion":
// after a verification the suffix past the rejection point is discarded from
// the caches and the next round starts from the last accepted token.  Hydra
// Guide, section "3. Tree KV-Cache Page Sizing": the discarded candidates are
// rolled back at once, without deallocation.  Here the verification's tree
// keys/values stay in their own buffers; committing the accepted path copies
// its m + 1 nodes' rows (root first) of every KV head to cache positions
// prefix_len[b] .. prefix_len[b] + m and advances prefix_len[b] by m + 1.  The
// rejected nodes are never copied, so rolling them back costs nothing.
//
// One CTA per sequence: warp 0 checks the path (root first, each node a
// child of the previous one, m <= max depth, the commit fits in Lmax); the CTA
// then copies the rows in 16-byte chunks and finally advances prefix_len[b],
// so no other CTA reads or writes that entry.  A sequence that fails a check is
// left unchanged and SPEC_EINVAL goes to the status word.  The paged form writes
// the same rows into pool blocks through the block table (Hydra Guide, "Hydra
// Production Engineering Checklist", item 3: the cache in pre-allocated static
// blocks), the layout the paged tree attention reads.
#include "common.cuh"

namespace spec {
namespace kv {

constexpr int kThreads = 256;

// Paged cache (table != NULL): cache position p of sequence b is row p % bs of pool
// block table[b, p / bs] (pool [num_blocks, Hkv, bs, D]); warp 0 also checks that
// every block the commit writes lies inside the pool and that the commit stays within
// max_blocks * bs positions.  Contiguous cache: the pool is [B, Hkv, Lmax, D], i.e.
// bs = Lmax and sequence b's only block is b.
__global__ void __launch_bounds__(kThreads) k_kv_commit(const uint4* __restrict__ k_tree, const uint4* __restrict__ v_tree,
                                                        uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                                                        int32_t* __restrict__ prefix_len,
                                                        const int32_t* __restrict__ accept_len,
                                                        const int32_t* __restrict__ accept_path, int path_stride,
                                                        const int32_t* __restrict__ parent, int T, int max_depth, int Hkv,
                                                        int Lmax, int row16, const int32_t* __restrict__ table,
                                                        int max_blocks, int bs, int num_blocks, void* ws) {
    const int b = blockIdx.x;
    __shared__ int s_path[SPEC_MAX_DEPTH + 1], s_blk[SPEC_MAX_DEPTH + 1];
    __shared__ int s_n, s_L;
    if (threadIdx.x < 32) {
        // warp 0 checks the path, lane i the i-th entry (max depth <= 16 < 32)
        const int lane = threadIdx.x;
        const int m = accept_len[b];
        const int L = prefix_len[b];
        const int64_t cap = table ? static_cast<int64_t>(max_blocks) * bs : Lmax;
        const bool len_ok = m >= 0 && m <= max_depth && L >= 0 && static_cast<int64_t>(L) + m + 1 <= cap;
        const bool mine = len_ok && lane <= m;
        const int node = mine ? accept_path[static_cast<size_t>(b) * path_stride + lane] : 0;
        const bool in_tree = node >= 0 && node < T;
        const int par = (mine && lane > 0 && in_tree) ? parent[node] : -1;
        const int prev = __shfl_up_sync(0xffffffffu, node, 1);
        int blk = b;
        if (mine && table) blk = table[static_cast<size_t>(b) * max_blocks + (L + lane) / bs];
        const bool blk_ok = !table || (blk >= 0 && blk < num_blocks);
        const bool ok_i = !mine || ((lane == 0 ? node == 0 : (in_tree && node > 0 && par == prev)) && blk_ok);
        const bool ok = len_ok && __all_sync(0xffffffffu, ok_i);
        if (mine) {
            s_path[lane] = node;
            s_blk[lane] = blk;
        }
        if (lane == 0) {
            if (!ok) flag_status(ws, SPEC_EINVAL);
            s_n = ok ? m + 1 : 0;
            s_L = L;
        }
    }
    __syncthreads();
    const int n = s_n, L = s_L;
    if (n == 0) return;
    const int rows = table ? bs : Lmax;   // rows per (block, head)
    // 16-byte chunks of K and V: each thread issues the loads of up to kBatch chunks
    // before their stores, so a sequence's rows are in flight together
    constexpr int kBatch = 8;
    const int per_head = n * row16;
    const int total = Hkv * per_head;
    for (int base = threadIdx.x; base < total; base += kThreads * kBatch) {
        uint4 kx[kBatch], vx[kBatch];
        size_t dst[kBatch];
#pragma unroll
        for (int q = 0; q < kBatch; ++q) {
            const int idx = base + q * kThreads;
            if (idx < total) {
                const int h = idx / per_head;
                const int rem = idx - h * per_head;
                const int i = rem / row16, c = rem - i * row16;
                const size_t src = ((static_cast<size_t>(b) * Hkv + h) * T + s_path[i]) * row16 + c;
                const int pos = table ? (L + i) % bs : L + i;
                dst[q] = ((static_cast<size_t>(s_blk[i]) * Hkv + h) * rows + pos) * row16 + c;
                kx[q] = k_tree[src];
                vx[q] = v_tree[src];
            }
        }
#pragma unroll
        for (int q = 0; q < kBatch; ++q) {
            if (base + q * kThreads < total) {
                k_cache[dst[q]] = kx[q];
                v_cache[dst[q]] = vx[q];
            }
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) prefix_len[b] = L + n;
}

}  // namespace kv
}  // namespace spec

using namespace spec;

extern "C" size_t tree_kv_commit_workspace_size(void) { return kWsHeader; }

namespace {
spec_status kv_commit_run(const void* k_tree, const void* v_tree, void* k_cache, void* v_cache, int32_t* prefix_len,
                          const int32_t* accept_len, const int32_t* accept_path, const spec_tree* tree, int32_t B,
                          int32_t Hkv, int32_t Lmax, int32_t D, spec_dtype dt, const int32_t* table, int32_t max_blocks,
                          int32_t bs, int32_t num_blocks, void* ws, size_t ws_bytes, cudaStream_t s) {
    spec_status st = check_tree(tree);
    if (st != SPEC_OK) return st;
    if (dt != SPEC_BF16 && dt != SPEC_F32) return fail(SPEC_EUNSUPPORTED, "dtype %d: only bf16 and fp32", static_cast<int>(dt));
    const int es = dt == SPEC_BF16 ? 2 : 4;
    if (B < 1 || B > 65535 || Hkv < 1 || Lmax < 1 || D < 1)
        return fail(SPEC_EINVAL, "B = %d (1..65535), Hkv = %d, Lmax = %d, D = %d must be positive", B, Hkv, Lmax, D);
    if ((static_cast<int64_t>(D) * es) % 16 != 0) return fail(SPEC_EINVAL, "D * element size = %d bytes: not a multiple of 16", D * es);
    const int row16 = D * es / 16;
    if (static_cast<int64_t>(Hkv) * (tree->max_depth + 1) * row16 > INT32_MAX)
        return fail(SPEC_EINVAL, "Hkv * (max depth + 1) * D too large");
    if (!k_tree || !v_tree || !k_cache || !v_cache || !prefix_len || !accept_len || !accept_path)
        return fail(SPEC_EINVAL, "no pointer argument may be NULL");
    if (!aligned16(k_tree) || !aligned16(v_tree) || !aligned16(k_cache) || !aligned16(v_cache))
        return fail(SPEC_EALIGN, "tree and cache buffers must be 16-byte aligned");
    if (!aligned4(prefix_len) || !aligned4(accept_len) || !aligned4(accept_path) || (table && !aligned4(table)))
        return fail(SPEC_EALIGN, "prefix_len, accept_len, accept_path and the block table must be 4-byte aligned");
    if (!ws || ws_bytes < kWsHeader) return fail(SPEC_EWORKSPACE, "workspace %zu bytes < %zu needed", ws_bytes, kWsHeader);
    if (!aligned16(ws)) return fail(SPEC_EALIGN, "workspace must be 16-byte aligned");
    SPEC_CUDA_TRY(reset_device_status(ws, s));
    SPEC_CUDA_TRY(launch("kv_commit", kv::k_kv_commit, dim3(B), dim3(kv::kThreads), 0, s,
                         static_cast<const uint4*>(k_tree), static_cast<const uint4*>(v_tree), static_cast<uint4*>(k_cache),
                         static_cast<uint4*>(v_cache), prefix_len, accept_len, accept_path, tree->max_depth + 1,
                         tree->parent, tree->T, tree->max_depth, Hkv, Lmax, row16, table, max_blocks, bs, num_blocks, ws));
    return SPEC_OK;
}
}  // namespace

extern "C" spec_status tree_kv_commit(const void* k_tree, const void* v_tree, void* k_cache, void* v_cache,
                                      int32_t* prefix_len, const int32_t* accept_len, const int32_t* accept_path,
                                      const spec_tree* tree, int32_t B, int32_t Hkv, int32_t Lmax, int32_t D,
                                      spec_dtype dt, void* ws, size_t ws_bytes, spec_stream_t s_) {
    clear_error();
    return kv_commit_run(k_tree, v_tree, k_cache, v_cache, prefix_len, accept_len, accept_path, tree, B, Hkv, Lmax, D,
                         dt, nullptr, 0, 0, 0, ws, ws_bytes, reinterpret_cast<cudaStream_t>(s_));
}

extern "C" spec_status tree_kv_commit_paged(const void* k_tree, const void* v_tree, void* k_pool, void* v_pool,
                                            int32_t num_blocks, const int32_t* block_table, int32_t max_blocks,
                                            int32_t block_size, int32_t* prefix_len, const int32_t* accept_len,
                                            const int32_t* accept_path, const spec_tree* tree, int32_t B, int32_t Hkv,
                                            int32_t D, spec_dtype dt, void* ws, size_t ws_bytes, spec_stream_t s_) {
    clear_error();
    if (num_blocks < 1 || max_blocks < 1 || block_size < 1)
        return fail(SPEC_EINVAL, "num_blocks = %d, max_blocks = %d, block_size = %d must be positive", num_blocks,
                    max_blocks, block_size);
    if (static_cast<int64_t>(max_blocks) * block_size > (1 << 22))
        return fail(SPEC_EINVAL, "max_blocks * block_size = %lld positions exceed 2^22",
                    static_cast<long long>(max_blocks) * block_size);
    if (!block_table) return fail(SPEC_EINVAL, "block_table must not be NULL");
    return kv_commit_run(k_tree, v_tree, k_pool, v_pool, prefix_len, accept_len, accept_path, tree, B, Hkv,
                         max_blocks * block_size, D, dt, block_table, max_blocks, block_size, num_blocks, ws, ws_bytes,
                         reinterpret_cast<cudaStream_t>(s_));
}
