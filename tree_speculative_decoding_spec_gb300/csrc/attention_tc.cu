// Tensor-core (tcgen05) path of tree attention.
//
// Hydra Guide, "Tree Attention Matrix with Topology-Aware Causal Masking":
// every tree node sees the cached prefix and its own ancestors; the ancestor
// sets arrive as one bit row per node and are applied to the scores in
// registers.
//
// One CTA = one (prefix split, KV head x 128-query-row block, sequence); the
// CTA holding the last non-empty prefix split of a sequence also takes the
// tree keys.  The query rows of a KV head are its g query heads x T nodes,
// contiguous in q [B, Hq, T, D], so one 2-D TMA box fetches them.  Eleven warps:
//   warp 8    TMA: the 128 x 128 Q tile once, then a 3-stage ring of 128-key
//             K and V tiles (128-byte swizzle), prefix tiles then tree tiles
//   warps 9, 10  MMA, one thread each: warp 9 + g issues the MMAs of the
//             tiles j with j % 2 == g -- S_j = Q K_j^T into TMEM score buffer g
//             (M 128, N 128, K 128, both operands in shared memory) and
//             O_g += P_j V_j (M 128, N 128, K 128) with P_j read from TMEM and
//             V as an MN-major shared-memory operand
//   warps 0-3 / 4-7: two softmax groups; group j % 2 owns tile j.  One thread
//             per query row reads S_j from TMEM, masks (prefix length,
//             ancestor bits), keeps its group's running maximum and sum in
//             base 2 (O is rescaled in TMEM only when the maximum grows by
//             more than 2^8) and writes P_j as bf16 pairs over the first 64
//             columns of its own score buffer.  At the end group 0 merges the
//             two groups' (max, sum, O): with a single split it writes out and
//             lse directly; otherwise the split's partial goes to HBM for the
//             combine kernel, or -- when the splits of a (head, row block,
//             sequence) run as one thread-block cluster -- it stays in the
//             CTA's own shared memory and is merged across the cluster over
//             distributed shared memory (see the end of the kernel).
// A thread's MMAs run in its issue order, so S_{j+2} may overwrite the buffer
// PV_j reads, and the completion of S_j implies that of PV_{j-2} (same thread);
// the two threads share only the K/V ring, whose stages free in tile order.
// Cache rows past the prefix length inside the last prefix tile are zeroed in
// shared memory before PV reads them (their scores are masked, and a stale
// non-finite value times a zero weight would still poison O).
// Waits are bounded (2 s); on expiry SPEC_ETIMEOUT goes to the status word and
// the CTA drains its own loads and MMAs before freeing TMEM.
#include <algorithm>

#include "attention_tc.cuh"
#include "tc.cuh"

namespace spec {
namespace tc {

constexpr int kARows = 128;        // query rows per CTA (MMA M)
constexpr int kAKeys = 128;        // keys per tile
constexpr int kAD = 128;           // head dim
constexpr int kAStages = 3;
// Landing barriers of the K/V ring: tile j signals k_full[j % kKFull].  The stages
// alternate between the two MMA threads (tile j belongs to thread j % 2), so with
// one barrier per stage a thread would wait on a phase whose predecessor the other
// thread consumed -- and a parity wait cannot tell a phase still open from one two
// phases back (a tile landing out of order would pass it early).  With 2 x kAStages
// barriers each belongs to one thread, which waits on every phase of it in order.
constexpr int kKFull = 2 * kAStages;
constexpr int kAPrefetch = 2;     // contiguous prefix tiles prefetched into L2 ahead of their load
constexpr int kAThreads = 352;
constexpr int kQBytes = 2 * kARows * 128;         // two 64-column halves of 128 rows
constexpr int kKVHalf = kAKeys * 128;             // one 64-column half of a 128-key tile
constexpr int kStageBytes = 4 * kKVHalf;          // K and V, two halves each
constexpr size_t kASmem = 1024 + kQBytes + kAStages * kStageBytes + 2048;
constexpr uint32_t kATmemCols = 512;              // S0 [0,128) S1 [128,256) O0 [256,384) O1 [384,512)
constexpr uint32_t kAO = 2 * kAKeys;              // first O column
constexpr int kFusedMaxSplits = 8;                // portable cluster size
constexpr int kFPStride = kAD + 4;                // floats per row of an on-chip partial: m, l, -, -, O[kAD]
static_assert(kASmem <= 232448, "shared memory of one CTA");

struct AttnTcParams {
    int T, g, Hq, Hkv, Lmax, words;
    int chunk, n_pre, n_rb;
    float scale_log2;
    const int32_t* prefix_len;
    const uint64_t* anc;
    float* part;
    void* ws;
    KvPages pg;
    int fused;          // cluster of the n_pre splits: merge on chip, write out / lse
    float* out;
    float* lse;
};

// Packed two-lane fp32 arithmetic (sm_100 family): one instruction for a pair of
// scores halves the softmax's FFMA and FADD count, and the 3-input max does the
// same for the row maximum.
__device__ __forceinline__ unsigned long long pk2(float a, float b) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void upk2(unsigned long long r, float& a, float& b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ unsigned long long ffma2(unsigned long long a, unsigned long long b, unsigned long long c) {
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ unsigned long long fadd2(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// The sequence of grid slot z: sequences in order of decreasing prefix length
// (ties to the lower index).  CTAs start in grid order, so the longest work
// starts first and the shorter fills in behind it as SMs free up
// (longest-processing-time-first); variable prefix lengths would otherwise
// leave a second wave led by a long sequence.  Each warp ranks up to 64
// sequences on its own (two per lane); larger batches keep the identity.
__device__ __forceinline__ int longest_first(const int32_t* __restrict__ prefix_len, int B, int z) {
    if (B <= 1 || B > 64) return z;
    const int lane = threadIdx.x & 31;
    int found = -1;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int i = lane + 32 * h;
        int rank = -1;
        if (i < B) {
            const int li = prefix_len[i];
            rank = 0;
            for (int j = 0; j < B; ++j) {
                const int lj = prefix_len[j];
                rank += (lj > li) || (lj == li && j < i);
            }
        }
        const unsigned hit = __ballot_sync(0xffffffffu, rank == z);
        if (hit) found = 32 * h + __ffs(hit) - 1;
    }
    return found < 0 ? z : found;
}

// Named barrier for the 256 softmax threads (warps 0-7).
__device__ __forceinline__ void softmax_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// kApart: every CTA's tiles fit in the ring at once (short prefixes); K and V of a stage then
// complete on separate barriers, so S_j starts as soon as K_j has landed.  In a long stream
// one barrier covers both (S_j waits for V_j too, which keeps V_j's shared-memory writes off
// S_j's operand reads); the two forms are separate instantiations so that neither carries
// the other's waits.
template <bool kApart>
__global__ void __launch_bounds__(kAThreads, 1) k_attn_tc(const __grid_constant__ CUtensorMap tmQ,
                                                          const __grid_constant__ CUtensorMap tmKc,
                                                          const __grid_constant__ CUtensorMap tmVc,
                                                          const __grid_constant__ CUtensorMap tmKt,
                                                          const __grid_constant__ CUtensorMap tmVt,
                                                          const AttnTcParams p) {
    const int c = blockIdx.x;
    const int kvh = blockIdx.y / p.n_rb, rb = blockIdx.y % p.n_rb;
    const int b = longest_first(p.prefix_len, gridDim.z, blockIdx.z);
    const int L = min(max(p.prefix_len[b], 0), p.Lmax);
    const int pre_begin = c * p.chunk;
    const int pre_end = min(L, pre_begin + p.chunk);
    const int n_pt = pre_end > pre_begin ? (pre_end - pre_begin + kAKeys - 1) / kAKeys : 0;
    const int n_pref = (L + p.chunk - 1) / p.chunk;          // non-empty prefix splits
    const bool has_tree = (c == max(n_pref - 1, 0));          // this split also takes the tree keys
    const bool direct = p.n_pre == 1;                         // one split: write out and lse here
    const int n_tt = has_tree ? (p.T + kAKeys - 1) / kAKeys : 0;
    const int n_tiles = n_pt + n_tt;
    if (n_tiles == 0 && !p.fused) return;   // whole CTA: nothing allocated yet (a fused one still merges)

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = smem;
    uint8_t* sKV = sQ + kQBytes;                       // stage s: K half0, K half1, V half0, V half1
    uint64_t* bars = reinterpret_cast<uint64_t*>(sKV + kAStages * kStageBytes);
    uint64_t* q_full = bars;
    uint64_t* k_full = bars + 1;                       // [j % kKFull] tile j's K (and V, unless kApart) landed
    uint64_t* v_full = k_full + kKFull;                // [stage] its V tile landed (kApart only)
    uint64_t* kv_empty = v_full + kAStages;            // [stage] PV of the stage's tile complete
    uint64_t* s_full = kv_empty + kAStages;            // [group]
    uint64_t* p_full = s_full + 2;                     // [group]
    uint64_t* o_final = p_full + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(o_final + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    float2* merge = reinterpret_cast<float2*>(reinterpret_cast<uint8_t*>(bars) + 256);   // [128] group 1's (m, l)
    static_assert((1 + kKFull + 2 * kAStages + 5) * 8 + 8 <= 256, "barriers and flags end before the merge buffer");

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int s = 0; s < kKFull; ++s) mbar_init(&k_full[s], 1);
        for (int s = 0; s < kAStages; ++s) {
            mbar_init(&v_full[s], 1);
            mbar_init(&kv_empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[i], 4);   // one arrival per softmax warp
        }
        mbar_init(o_final, 2);   // one commit from each MMA thread
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&tmQ);
        prefetch_tmap(&tmKc);
        prefetch_tmap(&tmVc);
        if (n_tt) {
            prefetch_tmap(&tmKt);
            prefetch_tmap(&tmVt);
        }
    }
    if (warp == 0) tmem_alloc(tmem_slot, kATmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    griddep_launch();   // the next kernel on the stream may start launching
    const int kvc_row0 = (b * p.Hkv + kvh) * p.Lmax + pre_begin;   // first prefix key of this split
    const int kvt_row0 = (b * p.Hkv + kvh) * p.T;                  // first tree key
    const int q_row0 = (b * p.Hq + kvh * p.g) * p.T + rb * kARows;
    int issued = 0;

    if (warp == 8) {
        if (lane == 0) {
            mbar_arrive_expect_tx(q_full, kQBytes);
            tma_load_2d(sQ, &tmQ, q_full, 0, q_row0);
            tma_load_2d(sQ + kARows * 128, &tmQ, q_full, 64, q_row0);
            // a stage frees once PV of its tile is complete
            for (int j = 0; j < n_tiles; ++j) {
                const int s = j % kAStages;
                const bool tree_tile = j >= n_pt;
                uint8_t* st = sKV + s * kStageBytes;
                // source rows of the tile's two 64-key halves
                int row_h[2];
                if (!tree_tile && p.pg.table) {
                    // paged prefix: each half lies inside one pool block (bs is a multiple of 64);
                    // keys past the prefix read the last used block (they are masked, and their
                    // V rows zeroed, by the softmax threads)
                    for (int hh = 0; hh < 2; ++hh) {
                        const int pos = pre_begin + j * kAKeys + hh * 64;
                        const int lb = min(pos / p.pg.bs, (L - 1) / p.pg.bs);
                        int blk = p.pg.table[static_cast<size_t>(b) * p.pg.max_blocks + lb];
                        if (blk < 0 || blk >= p.pg.num_blocks) {
                            flag_status(p.ws, SPEC_EINVAL);
                            blk = 0;
                        }
                        row_h[hh] = (blk * p.Hkv + kvh) * p.pg.bs + pos % p.pg.bs;
                    }
                } else {
                    row_h[0] = tree_tile ? kvt_row0 + (j - n_pt) * kAKeys : kvc_row0 + j * kAKeys;
                    row_h[1] = row_h[0] + 64;
                }
                // one 128-key box per 64-column half, or two 64-key boxes when paged
                auto load = [&](const CUtensorMap* mc, const CUtensorMap* mt, uint64_t* bar, uint8_t* dst) {
                    if (!tree_tile && p.pg.table) {
                        for (int hh = 0; hh < 2; ++hh) {
                            const int off = hh * (kKVHalf / 2);
                            tma_load_2d(dst + off, mc, bar, 0, row_h[hh]);
                            tma_load_2d(dst + kKVHalf + off, mc, bar, 64, row_h[hh]);
                        }
                    } else {
                        const CUtensorMap* m = tree_tile ? mt : mc;
                        tma_load_2d(dst, m, bar, 0, row_h[0]);
                        tma_load_2d(dst + kKVHalf, m, bar, 64, row_h[0]);
                    }
                };
                if (j >= kAStages && !mbar_wait_or_abort(&kv_empty[s], ((j / kAStages) - 1) & 1, abort_flag)) {
                    flag_status(p.ws, SPEC_ETIMEOUT);
                    *abort_flag = 1;
                    break;
                }
                uint64_t* kbar = &k_full[j % kKFull];
                uint64_t* vbar = kApart ? &v_full[s] : kbar;
                mbar_arrive_expect_tx(kbar, kApart ? 2 * kKVHalf : kStageBytes);
                load(&tmKc, &tmKt, kbar, st);
                if (kApart) mbar_arrive_expect_tx(vbar, 2 * kKVHalf);
                load(&tmVc, &tmVt, vbar, st + 2 * kKVHalf);
                issued = j + 1;
                // the prefix tile kAPrefetch tiles ahead heads for L2 now: the ring's lead
                // (its stages free up only as PV finishes) is shorter than a load's latency
                const int jp = j + kAPrefetch;
                if (kAPrefetch > 0 && jp < n_pt && !p.pg.table) {
                    const int rp = kvc_row0 + jp * kAKeys;
                    tma_prefetch_2d(&tmKc, 0, rp);
                    tma_prefetch_2d(&tmKc, 64, rp);
                    tma_prefetch_2d(&tmVc, 0, rp);
                    tma_prefetch_2d(&tmVc, 64, rp);
                }
            }
        }
        __syncwarp();
    } else if (warp == 9 || warp == 10) {
        // two MMA threads, one per softmax group: thread g issues S and PV of the tiles j with
        // j % 2 == g, so each group's MMAs stay in issue order (the buffer reuse below relies
        // on that) while one thread's waits and commits overlap the other's MMAs
        const int g = warp - 9;
        if (lane == 0) {
            const uint32_t idesc_s = idesc_bf16_f32(kARows, kAKeys);
            const uint32_t idesc_o = idesc_bf16_f32_bmn(kARows, kAD);
            // a descriptor's start-address field is the byte address / 16 in its low 14 bits;
            // offsets inside shared memory never carry out of it, so the descriptor of an
            // offset sub-tile is the base descriptor plus offset / 16
            const uint64_t qd = sdesc_k128(smem_u32(sQ));
            bool ok = mbar_wait_or_abort(q_full, 0, abort_flag);
            // this thread's landing barrier and phase for its next S (j = g, g + 2, ...), kept
            // as counters: no division on the issue path
            int kf = g;
            uint32_t kf_phase = 0;
            // S_j = Q K_j^T: K = 128 in 8 steps of 16 (two 64-column halves)
            auto issue_s = [&](int j) -> bool {
                const int s = j % kAStages;
                if (!mbar_wait_or_abort(&k_full[kf], kf_phase, abort_flag)) return false;
                kf += 2;
                if (kf >= kKFull) {
                    kf -= kKFull;
                    kf_phase ^= 1u;
                }
                tc_fence_after();
                const uint64_t kd = sdesc_k128(smem_u32(sKV + s * kStageBytes));
                const uint32_t dst = tmem + (j & 1) * kAKeys;
#pragma unroll
                for (int ks = 0; ks < kAD / 16; ++ks) {
                    const uint32_t off = (ks & 3) * 32;
                    mma_bf16(dst, qd + (((ks >> 2) * (kARows * 128) + off) >> 4), kd + (((ks >> 2) * kKVHalf + off) >> 4),
                             idesc_s, ks > 0 ? 1u : 0u);
                }
                mma_commit(&s_full[j & 1]);
                return true;
            };
            // S for the group's first tile, then per tile: PV_j, S_{j+2}
            if (ok && g < n_tiles) ok = issue_s(g);
            for (int j = g; ok && j < n_tiles; j += 2) {
                if (!mbar_wait_or_abort(&p_full[j & 1], (j >> 1) & 1, abort_flag)) { ok = false; break; }
                if constexpr (kApart) {
                    if (!mbar_wait_or_abort(&v_full[j % kAStages], 0, abort_flag)) { ok = false; break; }
                }
                tc_fence_after();
                // O_{j%2} += P_j V_j: K = 128 keys in 8 steps of 16.  P_j: bf16 pairs in the first
                // 64 columns of score buffer j % 2 (8 columns per step).  V is MN-major (d
                // contiguous): 64-wide d halves kKVHalf apart, 8-key atoms 1 KB apart.
                const uint32_t pa = tmem + (j & 1) * kAKeys;
                const uint64_t vd = sdesc_mn128(smem_u32(sKV + (j % kAStages) * kStageBytes + 2 * kKVHalf), kKVHalf, 1024);
                const uint32_t o = tmem + kAO + (j & 1) * kAD;
#pragma unroll
                for (int ks = 0; ks < kAKeys / 16; ++ks)
                    mma_bf16_ts(o, pa + ks * 8, vd + ((ks * 2048) >> 4), idesc_o,
                                (j >= 2 || ks > 0) ? 1u : 0u);
                mma_commit(&kv_empty[j % kAStages]);
                // in issue order after PV_j, so S_{j+2} may overwrite P_j
                if (j + 2 < n_tiles && !issue_s(j + 2)) { ok = false; break; }
            }
            if (!ok) {
                flag_status(p.ws, SPEC_ETIMEOUT);
                *abort_flag = 1;
            }
            mma_commit(o_final);
        }
        __syncwarp();
    } else {
        const int grp = warp >> 2;                         // softmax group: tiles j with j % 2 == grp
        const int r = (warp & 3) * 32 + lane;              // query row of this block = TMEM lane
        const int rg = rb * kARows + r;                    // row within the KV head's g*T rows
        const int node = rg % p.T;
        const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        const uint32_t s_col = grp * kAKeys;
        const uint32_t o_col = kAO + grp * kAD;
        const uint64_t* anc_row = p.anc + static_cast<size_t>(node) * p.words;
        float m_used = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = grp; j < n_tiles; j += 2) {
            // S_j complete also means PV_{j-2} (same O, same buffer) is complete
            ok = __all_sync(0xffffffffu, mbar_wait_or_abort(&s_full[grp], (j >> 1) & 1, abort_flag));
            if (!ok) break;
            tc_fence_after();
            uint32_t s0[32], s1[32], s2[32], s3[32];
            tmem_ld32(lane_base + s_col, s0);
            tmem_ld32(lane_base + s_col + 32, s1);
            tmem_ld32(lane_base + s_col + 64, s2);
            tmem_ld32(lane_base + s_col + 96, s3);
            tmem_ld_wait();
            auto sraw = [&](int e) -> uint32_t {
                return e < 32 ? s0[e] : e < 64 ? s1[e - 32] : e < 96 ? s2[e - 64] : s3[e - 96];
            };
            // raw scores (the scale is applied inside the exponent: scale > 0 keeps the order);
            // masking only on tree tiles and on a partial last prefix tile (tile-uniform branch)
            float sv[kAKeys];
            const bool tree_tile = j >= n_pt;
            const int nvalid = tree_tile ? min(kAKeys, p.T - (j - n_pt) * kAKeys)
                                         : min(kAKeys, pre_end - (pre_begin + j * kAKeys));
            if (!tree_tile && nvalid == kAKeys) {
#pragma unroll
                for (int e = 0; e < kAKeys; ++e) sv[e] = __uint_as_float(sraw(e));
            } else {
                uint64_t bits[2];
#pragma unroll
                for (int w = 0; w < 2; ++w) {
                    const int nv = min(max(nvalid - 64 * w, 0), 64);
                    bits[w] = nv >= 64 ? ~0ull : ((1ull << nv) - 1ull);
                }
                if (tree_tile) {   // only the node's ancestors (and itself)
                    const int w0 = 2 * (j - n_pt);
                    bits[0] &= anc_row[w0];
                    bits[1] &= (w0 + 1 < p.words) ? anc_row[w0 + 1] : 0ull;
                }
#pragma unroll
                for (int e = 0; e < kAKeys; ++e)
                    sv[e] = ((bits[e >> 6] >> (e & 63)) & 1ull) ? __uint_as_float(sraw(e)) : -INFINITY;
            }
            float mx[16];
#pragma unroll
            for (int e = 0; e < 16; ++e)
                mx[e] = fmax3(fmax3(sv[e], sv[e + 16], sv[e + 32]), fmax3(sv[e + 48], sv[e + 64], sv[e + 80]),
                              fmax3(sv[e + 96], sv[e + 112], -INFINITY));
            mx[0] = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmax3(mx[6], mx[7], mx[8]));
            mx[0] = fmax3(fmax3(mx[0], mx[9], mx[10]), fmax3(mx[11], mx[12], mx[13]), fmaxf(mx[14], mx[15]));
            const float tmax = mx[0] * p.scale_log2;   // base-2 units
            // lazy rescale: keep the old reference maximum unless the row max grew by > 2^8; the
            // TMEM accesses are warp-collective, so a warp rescales together (alpha = 1 for the rest)
            float m_new = m_used, alpha = 1.f;
            bool rescale = false;
            if (tmax > m_used + 8.f) {
                if (m_used != -INFINITY) {
                    rescale = true;
                    alpha = ex2(m_used - tmax);
                }
                m_new = tmax;
            }
            if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
                for (int cc = 0; cc < kAD / 16; ++cc) {
                    uint32_t o[16];
                    tmem_ld16(lane_base + o_col + cc * 16, o);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                    tmem_st16(lane_base + o_col + cc * 16, o);
                }
                l *= alpha;
            }
            m_used = m_new;
            // P = 2^(scale * s - m_used) in bf16 (one packed FFMA per pair of scores, one ex2 per
            // score), written over the first 64 columns of this group's score buffer; row sum in
            // fp32 over 4 partials of packed adds
            const float nmref = m_used == -INFINITY ? 0.f : -m_used;
            float ps[4];
#pragma unroll
            for (int qc = 0; qc < 4; ++qc) {
                uint32_t packed[16];
                unsigned long long acc2 = pk2(0.f, 0.f);
                const unsigned long long sc2 = pk2(p.scale_log2, p.scale_log2), nm2 = pk2(nmref, nmref);
#pragma unroll
                for (int h2 = 0; h2 < 16; ++h2) {
                    const int e0 = qc * 32 + 2 * h2;
                    float x0, x1;
                    upk2(ffma2(pk2(sv[e0], sv[e0 + 1]), sc2, nm2), x0, x1);
                    const float a0 = ex2(x0), a1 = ex2(x1);
                    acc2 = fadd2(acc2, pk2(a0, a1));
                    const __nv_bfloat162 pr = __floats2bfloat162_rn(a0, a1);   // .x (lower key) low
                    packed[h2] = *reinterpret_cast<const uint32_t*>(&pr);
                }
                float acc0, acc1;
                upk2(acc2, acc0, acc1);
                ps[qc] = acc0 + acc1;
                tmem_st16(lane_base + s_col + qc * 16, packed);
            }
            l += (ps[0] + ps[1]) + (ps[2] + ps[3]);
            if (!tree_tile && nvalid < kAKeys) {
                // zero the V rows past the prefix (both 64-column halves) once they have landed
                // and before PV_j reads them
                if constexpr (kApart) {
                    ok = __all_sync(0xffffffffu, mbar_wait_or_abort(&v_full[j % kAStages], 0, abort_flag));
                    if (!ok) break;
                }
                uint8_t* sv_tile = sKV + (j % kAStages) * kStageBytes + 2 * kKVHalf;
                const int r_in = (warp & 3) * 32 + lane;
                for (int i = r_in; i < (kAKeys - nvalid) * 16; i += kARows) {
                    const int row = nvalid + (i >> 4);
                    *reinterpret_cast<uint4*>(sv_tile + ((i >> 3) & 1) * kKVHalf + row * 128 + (i & 7) * 16) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async_smem();
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[grp]);
        }
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait_or_abort(o_final, 0, abort_flag));
        if (!ok) {
            flag_status(p.ws, SPEC_ETIMEOUT);
            *abort_flag = 1;
        }
        if (grp == 1) merge[r] = make_float2(m_used, l);
        softmax_sync();
        if (grp == 0 && !*abort_flag) {
            tc_fence_after();
            // merge the two groups: (m, l, O) = rescaled sums of (m0, l0, O0) and (m1, l1, O1)
            const float2 g1 = merge[r];
            const float m = fmaxf(m_used, g1.x);
            const float a0 = m_used == -INFINITY ? 0.f : ex2(m_used - m);
            const float a1 = g1.x == -INFINITY ? 0.f : ex2(g1.x - m);
            const bool valid = rg < p.T * p.g;
            const size_t out_row = (static_cast<size_t>(b) * p.Hq + kvh * p.g + rg / p.T) * p.T + rg % p.T;
            const float lsum = a0 * l + a1 * g1.y;
            float* dst = nullptr;   // (m, l, -, -, O[kAD]) partial at dst, or the output row itself when direct
            int o_off = 4;          // first O float at dst
            float scale_o = 1.f;
            if (p.fused) {   // this CTA's partial stays in its own shared memory (the drained K/V ring)
                dst = reinterpret_cast<float*>(sKV) + r * kFPStride;
            } else if (valid && direct) {
                dst = p.out + out_row * kAD;
                o_off = 0;
                scale_o = 1.f / lsum;
                if (p.lse) p.lse[out_row] = (m + log2f(lsum)) * 0.6931471805599453f;
            } else if (valid) {
                dst = p.part + (out_row * (p.n_pre + 1) + c) * (kAD + 4);
            }
            if (dst && !direct) {
                dst[0] = m;
                dst[1] = lsum;
            }
#pragma unroll 1
            for (int cc = 0; cc < kAD / 32; ++cc) {
                uint32_t o0[32], o1[32];
                tmem_ld32(lane_base + kAO + cc * 32, o0);
                tmem_ld32(lane_base + kAO + kAD + cc * 32, o1);
                tmem_ld_wait();
                if (dst) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        float v[4];
#pragma unroll
                        for (int t = 0; t < 4; ++t) {
                            const float x0 = a0 * __uint_as_float(o0[4 * e + t]);
                            v[t] = (a1 != 0.f ? x0 + a1 * __uint_as_float(o1[4 * e + t]) : x0) * scale_o;   // group 1 may own no tile
                        }
                        *reinterpret_cast<float4*>(dst + o_off + cc * 32 + 4 * e) = make_float4(v[0], v[1], v[2], v[3]);
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (*abort_flag) {
        // a wait ran out: let this CTA's own loads and MMAs land before releasing memory
        if (warp == 8 && lane == 0) {
            for (int j = max(0, issued - kAStages); j < issued; ++j) {
                mbar_wait(&k_full[j % kKFull], (j / kKFull) & 1, 100000000ull);
                if (kApart) mbar_wait(&v_full[j % kAStages], 0, 100000000ull);
            }
            mbar_wait(q_full, 0, 100000000ull);
        }
        if ((warp == 9 || warp == 10) && lane == 0) mbar_wait(o_final, 0, 100000000ull);
    }
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kATmemCols);
    }
    if (p.fused) {
        // The n_pre splits of this (KV head, row block, sequence) are one cluster, each
        // holding its (m, l, O) partial in shared memory (an aborted CTA publishes an empty
        // one: its own loads have landed by now).  After the cluster barrier CTA c merges
        // rows c, c + n, ... over every partial through distributed shared memory and
        // writes out = O / l and lse; a second barrier keeps each partial alive until
        // every peer has read it.  Every CTA reaches both barriers, also after a timeout.
        float* fpart = reinterpret_cast<float*>(sKV);
        if (*abort_flag && threadIdx.x < kARows) {
            fpart[threadIdx.x * kFPStride] = -INFINITY;
            fpart[threadIdx.x * kFPStride + 1] = 0.f;
        }
        cluster_sync();
        const int nc = static_cast<int>(gridDim.x);
        const int cr = static_cast<int>(cluster_ctarank());
        const uint32_t fbase = smem_u32(fpart);
        for (int r = cr + nc * warp; r < kARows; r += nc * (kAThreads / 32)) {
            const int rg = rb * kARows + r;
            if (rg >= p.T * p.g) break;   // rows only grow along the loop
            const uint32_t roff = fbase + static_cast<uint32_t>(r * kFPStride) * 4u;
            // every split's m, then every non-empty split's l and O chunk, each batch of
            // loads issued together
            float mj[kFusedMaxSplits], lj[kFusedMaxSplits];
            float4 vj[kFusedMaxSplits];
            float M = -INFINITY;
#pragma unroll
            for (int j = 0; j < kFusedMaxSplits; ++j) {
                mj[j] = j < nc ? dsmem_ld_f32(dsmem_map(roff, j)) : -INFINITY;
                M = fmaxf(M, mj[j]);
            }
#pragma unroll
            for (int j = 0; j < kFusedMaxSplits; ++j) {
                lj[j] = 0.f;
                vj[j] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (mj[j] != -INFINITY) {   // an empty split's O is never read
                    const uint32_t pj = dsmem_map(roff, j);
                    lj[j] = dsmem_ld_f32(pj + 4u);
                    vj[j] = dsmem_ld_f32x4(pj + 16u + 16u * lane);
                }
            }
            float lsum = 0.f;
            float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int j = 0; j < kFusedMaxSplits; ++j) {
                const float w = mj[j] == -INFINITY ? 0.f : exp2f(mj[j] - M);
                lsum += w * lj[j];
                o.x += w * vj[j].x;
                o.y += w * vj[j].y;
                o.z += w * vj[j].z;
                o.w += w * vj[j].w;
            }
            const int hl = rg / p.T, i = rg % p.T;
            const size_t row = (static_cast<size_t>(b) * p.Hq + kvh * p.g + hl) * p.T + i;
            const float inv = 1.f / lsum;
            *reinterpret_cast<float4*>(p.out + row * kAD + 4 * lane) = make_float4(o.x * inv, o.y * inv, o.z * inv, o.w * inv);
            if (p.lse && lane == 0) p.lse[row] = (M + log2f(lsum)) * 0.6931471805599453f;
        }
        cluster_sync();
    }
}

// ---------------------------------------------------------------- host

bool attn_tc_supported(int rows_per_kv_head, int D) {
    if (D != kAD || rows_per_kv_head < 64) return false;
    CUtensorMap probe;
    alignas(256) static const uint16_t dummy[kAD * 64] = {};
    // tensor-map encoding must be available (driver entry point); the probe map is never used
    return make_tmap_bf16_2d(&probe, dummy, 64, kAD, kAD, 64) == cudaSuccess;
}

// Clusters of n CTAs of k_attn_tc that the current device holds at once (0 when
// unknown, e.g. without a device), cached per device and cluster size.
static int max_active_clusters(int n) {
    static int cache[64][kFusedMaxSplits + 1];   // 0: not asked yet, -1: unavailable
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64 || n < 1 || n > kFusedMaxSplits) {
        cudaGetLastError();
        return 0;
    }
    int& c = cache[dev][n];
    if (c == 0) {
        int v = 0;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(n, 1, 1);
        cfg.blockDim = dim3(kAThreads);
        cfg.dynamicSmemBytes = kASmem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = n;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaFuncSetAttribute(k_attn_tc<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kASmem) != cudaSuccess ||
            cudaOccupancyMaxActiveClusters(&v, k_attn_tc<false>, &cfg) != cudaSuccess) {
            cudaGetLastError();
            v = 0;
        }
        c = v > 0 ? v : -1;
    }
    return c > 0 ? c : 0;
}

// Prefix splits: one CTA per (split, KV head x row block, sequence); the last
// non-empty split of each sequence also takes the tree keys.  Pick the split
// count minimising an estimated makespan -- waves of one CTA per SM times the
// longest CTA (its prefix tiles, the tree tiles, ~4 tiles of fixed cost: setup,
// the first loads, the epilogue), plus ~14 tiles for the combine kernel when the
// splits cannot merge on chip -- ties to fewer splits (less partial traffic).
// Merging on chip needs every cluster of the n splits resident at once.
constexpr int kPlanFixedTiles = 4;
constexpr int kPlanCombineTiles = 14;

AttnTcPlan attn_tc_plan(int B, int Hq, int Hkv, int T, int Lmax, int D, int sm_count) {
    AttnTcPlan p;
    const int g = Hq / Hkv;
    p.n_rb = (T * g + kARows - 1) / kARows;
    const int64_t base = static_cast<int64_t>(B) * Hkv * p.n_rb;
    const int tiles = (Lmax + kAKeys - 1) / kAKeys;
    const int tree_tiles = (T + kAKeys - 1) / kAKeys;
    auto fusable = [&](int n) { return n > 1 && n <= kFusedMaxSplits && base <= max_active_clusters(n); };
    int64_t best_cost = INT64_MAX;
    int best = 1;
    for (int n = 1; n <= std::min(tiles, 64); ++n) {
        const int per = (tiles + n - 1) / n;
        const int64_t waves = (base * n + sm_count - 1) / sm_count;
        const int64_t cost = waves * (per + tree_tiles + kPlanFixedTiles) + ((n > 1 && !fusable(n)) ? kPlanCombineTiles : 0);
        if (cost < best_cost) {
            best_cost = cost;
            best = n;
        }
    }
    p.chunk = static_cast<int>(round_up((Lmax + best - 1) / best, kAKeys));
    p.n_pre = (Lmax + p.chunk - 1) / p.chunk;
    // merge on chip only when every cluster is resident at once: a cluster starts only when
    // n_pre SMs of one GPC are free together, so a second wave of clusters leaves SMs idle
    // (32K prefix, 96 clusters of 3: 203 -> 296 us), and the one-split plans (a cluster of
    // one) write their output directly anyway
    p.fused = fusable(p.n_pre);
    // partial layout shared with the CUDA-core path: n_pre + 1 slots per row (the last unused
    // here); none with a single split or an on-chip merge
    p.part_bytes = (p.n_pre == 1 || p.fused)
                       ? 0 : sizeof(float) * static_cast<size_t>(B) * Hq * T * (p.n_pre + 1) * (D + 4);
    return p;
}

spec_status attn_tc_run(const AttnTcPlan& pl, const __nv_bfloat16* q, const __nv_bfloat16* kc, const __nv_bfloat16* vc,
                        const int32_t* prefix_len, const __nv_bfloat16* kt, const __nv_bfloat16* vt,
                        const spec_tree* tree, int B, int Hq, int Hkv, int Lmax, float scale, float* part, float* out,
                        float* lse, void* ws, cudaStream_t s, const KvPages& pg) {
    const int T = tree->T;
    CUtensorMap tq, tkc, tvc, tkt, tvt;
    SPEC_CUDA_TRY(make_tmap_bf16_2d(&tq, q, static_cast<uint64_t>(B) * Hq * T, kAD, kAD, kARows));
    if (pg.table) {   // pool rows, boxes of 64 (half a tile: one block holds it)
        SPEC_CUDA_TRY(make_tmap_bf16_2d(&tkc, kc, static_cast<uint64_t>(pg.num_blocks) * Hkv * pg.bs, kAD, kAD, 64));
        SPEC_CUDA_TRY(make_tmap_bf16_2d(&tvc, vc, static_cast<uint64_t>(pg.num_blocks) * Hkv * pg.bs, kAD, kAD, 64));
    } else {
        SPEC_CUDA_TRY(make_tmap_bf16_2d(&tkc, kc, static_cast<uint64_t>(B) * Hkv * Lmax, kAD, kAD, kAKeys));
        SPEC_CUDA_TRY(make_tmap_bf16_2d(&tvc, vc, static_cast<uint64_t>(B) * Hkv * Lmax, kAD, kAD, kAKeys));
    }
    SPEC_CUDA_TRY(make_tmap_bf16_2d(&tkt, kt, static_cast<uint64_t>(B) * Hkv * T, kAD, kAD, kAKeys));
    SPEC_CUDA_TRY(make_tmap_bf16_2d(&tvt, vt, static_cast<uint64_t>(B) * Hkv * T, kAD, kAD, kAKeys));
    AttnTcParams p{};
    p.T = T;
    p.g = Hq / Hkv;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.Lmax = Lmax;
    p.words = tree->words;
    p.chunk = pl.chunk;
    p.n_pre = pl.n_pre;
    p.n_rb = pl.n_rb;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.prefix_len = prefix_len;
    p.anc = tree->anc;
    p.part = part;
    p.ws = ws;
    p.pg = pg;
    p.fused = pl.fused ? 1 : 0;
    p.out = out;
    p.lse = lse;
    // every CTA's tiles (its prefix chunk, the tree tiles) fit in the ring at once
    const bool apart = pl.chunk / kAKeys + (T + kAKeys - 1) / kAKeys <= kAStages;
    auto kern = apart ? k_attn_tc<true> : k_attn_tc<false>;
    SPEC_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kASmem));
    if (pl.fused)
        SPEC_CUDA_TRY(launch_cluster("attn_tc", kern, dim3(pl.n_pre, Hkv * pl.n_rb, B), dim3(kAThreads), kASmem, s,
                                     false, dim3(pl.n_pre, 1, 1), tq, tkc, tvc, tkt, tvt, p));
    else
        SPEC_CUDA_TRY(launch("attn_tc", kern, dim3(pl.n_pre, Hkv * pl.n_rb, B), dim3(kAThreads), kASmem, s, tq,
                             tkc, tvc, tkt, tvt, p));
    return SPEC_OK;
}

}  // namespace tc
}  // namespace spec
