// Non-causal multi-head softmax attention of the DiT block on the tcgen05
// tensor cores, one request at a time (requests never attend to each other).
//
// qkv bf16 [R*T, 3h]: q | k | v column groups, head j at columns j*d of each.
// o   bf16 [R*T, h] : head j at columns j*d.
// O = softmax(Q K^T / sqrt(d)) V: fp32 logits in TMEM, fp32 online softmax,
// softmax weights rounded to bf16 for the P.V product, fp32 accumulation.
//
// One CTA = 128 query rows of one (request, head), 6 warps:
//   warp 0     TMA producer: Q once, then 128-key K and V tiles into a
//              STAGES-deep ring (3-D tensor map over [R, T, 3h], so a tile
//              never reaches into the next request: rows past T read zero);
//   warp 1     allocates TMEM (two 128-column S buffers + d columns of O);
//              lane 0 issues S_j = Q K_j^T (both operands K-major) into S
//              buffer j%2 and O += P_j V_j (P K-major from shared memory, V
//              MN-major straight from its TMA tile);
//   warps 2-5  softmax, one query row per thread (warp w owns TMEM lanes
//              32*(w%4)..+31): tcgen05.ld of the S row, keys past T masked to
//              -inf, running max m and sum l, P = exp2(S*c - m) written to
//              shared memory in the 128-byte-swizzled K-major layout the MMA
//              reads.  The running max is raised lazily - only when a row's
//              max grows by more than 2^8 - and O in TMEM is rescaled then;
//              otherwise P may reach 2^8, which fp32 and bf16 represent with
//              their usual relative precision, and O / l is the same softmax.
//              Finally O / l is written out as bf16.
// S is double-buffered so the next QK^T runs while this tile's softmax does.
// tcgen05.ld/st are warp-collective, so every branch around them is made
// uniform across the warp (__any_sync / __all_sync).  Every wait is bounded;
// on expiry the CTA records a code, drains its own copies and MMAs, frees
// TMEM and returns.
#include "dlo_device.cuh"
#include "dlo_internal.h"

namespace dlo {

namespace {

constexpr int kAttBM = 128;   // query rows per CTA
constexpr int kAttBN = 128;   // keys per tile
constexpr int kAttThreads = 192;
constexpr int kTileBytes = 128 * 128;  // one 128-row x 64-col bf16 box = 16 KB
constexpr float kLazyRescale = 8.0f;   // log2 units

template <int D>
struct AttCfg {
    static constexpr int kChunks = D / 64;                  // 64-wide column chunks of a head
    static constexpr int kQBytes = kChunks * kTileBytes;    // Q tile
    static constexpr int kKVBytes = kChunks * kTileBytes;   // one K (or V) tile
    static constexpr int kPBytes = 2 * kTileBytes;          // 128 x 128 bf16 P tile
    static constexpr int kStages = D == 64 ? 3 : 2;
    static constexpr int kSmem = kQBytes + 2 * kStages * kKVBytes + 2 * kPBytes;
    static constexpr int kSmemAlloc = kSmem + 1024 + 256;
    static constexpr uint32_t kTmemCols = 512;              // S0 | S1 | O
    static constexpr uint32_t kOCol = 256;
};

}  // namespace

enum : int {
    KERR_ATT_PRODUCER = 0x201,
    KERR_ATT_MMA = 0x202,
    KERR_ATT_SOFTMAX = 0x203,
    KERR_ATT_DRAIN = 0x204,
};

template <int D>
__global__ void __launch_bounds__(kAttThreads, 1)
    attention_fwd_tcgen05(const __grid_constant__ CUtensorMap tm, int T, int H, uint16_t* __restrict__ o,
                          float scale_log2, int* err) {
    using Cfg = AttCfg<D>;
    constexpr int ST = Cfg::kStages;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = smem;
    uint8_t* sK = sQ + Cfg::kQBytes;               // stage s at sK + s*kKVBytes
    uint8_t* sV = sK + ST * Cfg::kKVBytes;
    uint8_t* sP = sV + ST * Cfg::kKVBytes;         // buffer b at sP + b*kPBytes
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + Cfg::kSmem);
    uint64_t* q_full = bar;
    uint64_t* k_full = bar + 1;
    uint64_t* k_empty = k_full + ST;
    uint64_t* v_full = k_empty + ST;
    uint64_t* v_empty = v_full + ST;
    uint64_t* s_full = v_empty + ST;   // [2]
    uint64_t* p_full = s_full + 2;     // [2]
    uint64_t* o_done = p_full + 2;     // [2]
    uint64_t* drain = o_done + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q0 = blockIdx.x * kAttBM;
    const int head = blockIdx.y;
    const int req = blockIdx.z;
    const int h = H * D;
    const int n_kv = (T + kAttBN - 1) / kAttBN;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int s = 0; s < ST; ++s) {
            mbar_init(&k_full[s], 1);
            mbar_init(&k_empty[s], 1);
            mbar_init(&v_full[s], 1);
            mbar_init(&v_empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&s_full[b], 1);
            mbar_init(&p_full[b], 128);
            mbar_init(&o_done[b], 1);
        }
        mbar_init(drain, 1);
        fence_mbarrier_init();
        tma_prefetch_desc(&tm);
    }
    if (warp == 1) tmem_alloc(tmem_slot, Cfg::kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer
            long issued_k = 0, issued_v = 0;
            mbar_arrive_expect_tx(q_full, Cfg::kQBytes);
            for (int c = 0; c < Cfg::kChunks; ++c)
                tma_load_3d(sQ + c * kTileBytes, &tm, head * D + c * 64, q0, req, q_full);
            for (int j = 0; j < n_kv; ++j) {
                const int s = j % ST;
                const uint32_t ph = (uint32_t)((j / ST) & 1);
                if (!mbar_wait_bounded(&k_empty[s], ph ^ 1u, err, KERR_ATT_PRODUCER)) break;
                mbar_arrive_expect_tx(&k_full[s], Cfg::kKVBytes);
                for (int c = 0; c < Cfg::kChunks; ++c)
                    tma_load_3d(sK + s * Cfg::kKVBytes + c * kTileBytes, &tm, h + head * D + c * 64, j * kAttBN, req,
                                &k_full[s]);
                ++issued_k;
                if (!mbar_wait_bounded(&v_empty[s], ph ^ 1u, err, KERR_ATT_PRODUCER)) break;
                mbar_arrive_expect_tx(&v_full[s], Cfg::kKVBytes);
                for (int c = 0; c < Cfg::kChunks; ++c)
                    tma_load_3d(sV + s * Cfg::kKVBytes + c * kTileBytes, &tm, 2 * h + head * D + c * 64, j * kAttBN,
                                req, &v_full[s]);
                ++issued_v;
            }
            // every copy started here lands before the CTA exits
            mbar_wait_bounded(q_full, 0, err, KERR_ATT_DRAIN);
            for (long j = issued_k > ST ? issued_k - ST : 0; j < issued_k; ++j)
                mbar_wait_bounded(&k_full[j % ST], (uint32_t)((j / ST) & 1), err, KERR_ATT_DRAIN);
            for (long j = issued_v > ST ? issued_v - ST : 0; j < issued_v; ++j)
                mbar_wait_bounded(&v_full[j % ST], (uint32_t)((j / ST) & 1), err, KERR_ATT_DRAIN);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer
            constexpr uint32_t idesc_s = umma_idesc_bf16_f32(kAttBM, kAttBN);
            constexpr uint32_t idesc_pv = umma_idesc_bf16_f32(kAttBM, D) | (1u << 16);  // B (= V) MN-major
            const uint32_t q_addr = smem_u32(sQ);
            bool ok = mbar_wait_bounded(q_full, 0, err, KERR_ATT_MMA);
            auto issue_s = [&](int j) -> bool {
                const int s = j % ST;
                if (!mbar_wait_bounded(&k_full[s], (uint32_t)((j / ST) & 1), err, KERR_ATT_MMA)) return false;
                tc_fence_after();
                const uint32_t k_addr = smem_u32(sK + s * Cfg::kKVBytes);
                const uint32_t d_tmem = tmem + (uint32_t)((j & 1) * kAttBN);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (uint32_t)((kk >> 2) * kTileBytes + (kk & 3) * 32);
                    umma_bf16(d_tmem, umma_desc_sw128(q_addr + off), umma_desc_sw128(k_addr + off), idesc_s, kk > 0);
                }
                umma_commit(&k_empty[s]);
                umma_commit(&s_full[j & 1]);
                return true;
            };
            if (ok) ok = issue_s(0);
            if (ok && n_kv > 1) ok = issue_s(1);
            for (int j = 0; j < n_kv && ok; ++j) {
                const int b = j & 1;
                if (!mbar_wait_bounded(&p_full[b], (uint32_t)((j >> 1) & 1), err, KERR_ATT_MMA)) break;
                const int s = j % ST;
                if (!mbar_wait_bounded(&v_full[s], (uint32_t)((j / ST) & 1), err, KERR_ATT_MMA)) break;
                tc_fence_after();
                const uint32_t p_addr = smem_u32(sP + b * Cfg::kPBytes);
                const uint32_t v_addr = smem_u32(sV + s * Cfg::kKVBytes);
#pragma unroll
                for (int kk = 0; kk < kAttBN / 16; ++kk) {
                    const uint32_t poff = (uint32_t)((kk >> 2) * kTileBytes + (kk & 3) * 32);
                    umma_bf16(tmem + Cfg::kOCol, umma_desc_sw128(p_addr + poff),
                              umma_desc_sw128_mn(v_addr + (uint32_t)(kk * 2048), kTileBytes), idesc_pv,
                              (j > 0 || kk > 0) ? 1u : 0u);
                }
                umma_commit(&v_empty[s]);
                umma_commit(&o_done[b]);
                if (j + 2 < n_kv) ok = issue_s(j + 2);
            }
            umma_commit(drain);
            mbar_wait_bounded(drain, 0, err, KERR_ATT_DRAIN);
        }
    } else {
        // ---------------- softmax warpgroup (warps 2..5); all control flow
        // that encloses a tcgen05.ld/st is uniform across the warp.
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        const unsigned FULL = 0xffffffffu;
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < n_kv; ++j) {
            const int b = j & 1;
            ok = __all_sync(FULL, mbar_wait_bounded(&s_full[b], (uint32_t)((j >> 1) & 1), err, KERR_ATT_SOFTMAX));
            if (!ok) break;
            tc_fence_after();
            uint32_t sr[kAttBN];
#pragma unroll
            for (int c = 0; c < kAttBN / 32; ++c)
                tmem_ld_32x32b_x32_nowait(tmem + lane_base + (uint32_t)(b * kAttBN + c * 32), sr + c * 32);
            tmem_ld_wait();
            float t[kAttBN];
            const int valid = T - j * kAttBN;  // keys of this tile that exist
            float mx = -INFINITY;
#pragma unroll
            for (int i = 0; i < kAttBN; ++i) {
                t[i] = (i < valid) ? __uint_as_float(sr[i]) * scale_log2 : -INFINITY;
                mx = fmaxf(mx, t[i]);
            }
            if (j == 0) {
                m = mx;
            } else {
                // Raise this row's running max only if it grew by more than 2^8.
                const bool raise = mx > m + kLazyRescale;
                if (__any_sync(FULL, raise)) {
                    // The whole warp rescales its O rows (alpha = 1 for rows that keep
                    // their max) once PV_{j-1} has landed in TMEM.
                    const float alpha = raise ? exp2f(m - mx) : 1.0f;
                    if (raise) {
                        m = mx;
                        l *= alpha;
                    }
                    const int pb = (j - 1) & 1;
                    ok = __all_sync(FULL, mbar_wait_bounded(&o_done[pb], (uint32_t)(((j - 1) >> 1) & 1), err,
                                                            KERR_ATT_SOFTMAX));
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t orow[32];
                        const uint32_t oaddr = tmem + lane_base + Cfg::kOCol + (uint32_t)(c * 32);
                        tmem_ld_32x32b_x32_nowait(oaddr, orow);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i) orow[i] = __float_as_uint(__uint_as_float(orow[i]) * alpha);
                        tmem_st_32x32b_x32(oaddr, orow);
                    }
                    tmem_st_wait();
                }
            }
            // P buffer b was last read by PV_{j-2}
            if (j >= 2) {
                ok = __all_sync(FULL, mbar_wait_bounded(&o_done[b], (uint32_t)(((j - 2) >> 1) & 1), err,
                                                        KERR_ATT_SOFTMAX));
                if (!ok) break;
            }
            float rs = 0.f;
            uint8_t* prow = sP + b * Cfg::kPBytes + (row >> 3) * 1024 + (row & 7) * 128;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    float p[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        p[e] = exp2f(t[c * 64 + u * 8 + e] - m);
                        rs += p[e];
                    }
                    uint4 w;
                    w.x = pack_bf16x2(p[0], p[1]);
                    w.y = pack_bf16x2(p[2], p[3]);
                    w.z = pack_bf16x2(p[4], p[5]);
                    w.w = pack_bf16x2(p[6], p[7]);
                    *reinterpret_cast<uint4*>(prow + c * kTileBytes + ((u ^ (row & 7)) << 4)) = w;
                }
            }
            l += rs;
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&p_full[b]);
        }
        // O / l for this row, after the last P.V product
        if (ok) ok = __all_sync(FULL, mbar_wait_bounded(&o_done[(n_kv - 1) & 1], (uint32_t)(((n_kv - 1) >> 1) & 1),
                                                        err, KERR_ATT_SOFTMAX));
        if (ok) {
            tc_fence_after();
            const float inv = 1.f / l;
            const int t_row = q0 + row;
            uint16_t* orow = o + ((size_t)req * T + t_row) * h + head * D;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t v[32];
                tmem_ld_32x32b_x32_nowait(tmem + lane_base + Cfg::kOCol + (uint32_t)(c * 32), v);
                tmem_ld_wait();
                if (t_row < T) {
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        uint4 w;
                        w.x = pack_bf16x2(__uint_as_float(v[8 * g + 0]) * inv, __uint_as_float(v[8 * g + 1]) * inv);
                        w.y = pack_bf16x2(__uint_as_float(v[8 * g + 2]) * inv, __uint_as_float(v[8 * g + 3]) * inv);
                        w.z = pack_bf16x2(__uint_as_float(v[8 * g + 4]) * inv, __uint_as_float(v[8 * g + 5]) * inv);
                        w.w = pack_bf16x2(__uint_as_float(v[8 * g + 6]) * inv, __uint_as_float(v[8 * g + 7]) * inv);
                        *reinterpret_cast<uint4*>(orow + c * 32 + 8 * g) = w;
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, Cfg::kTmemCols);
    }
}

template <int D>
static int launch_attention_t(const uint16_t* qkv, int R, int T, int H, uint16_t* o, int* err, cudaStream_t st) {
    using Cfg = AttCfg<D>;
    static bool configured[64] = {};
    int dev = 0;
    DLO_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64) return set_error(DLO_ERR_INVALID_ARG, "device index %d out of range", dev);
    if (!configured[dev]) {
        DLO_CUDA_TRY(cudaFuncSetAttribute(attention_fwd_tcgen05<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          Cfg::kSmemAlloc));
        configured[dev] = true;
    }
    CUtensorMap tm;
    const uint64_t h = (uint64_t)H * D;
    int rc = encode_tmap_bf16_3d(&tm, qkv, 3 * h, (uint64_t)T, (uint64_t)R, 128);
    if (rc) return rc;
    const float scale_log2 = 1.4426950408889634f / sqrtf((float)D);
    dim3 grid((T + kAttBM - 1) / kAttBM, H, R);
    attention_fwd_tcgen05<D><<<grid, kAttThreads, Cfg::kSmemAlloc, st>>>(tm, T, H, o, scale_log2, err);
    DLO_CUDA_TRY(cudaGetLastError());
    return DLO_OK;
}

int launch_attention(const uint16_t* qkv, int R, int T, int H, int d, uint16_t* o, int* err, cudaStream_t st) {
    if (!qkv || !o || !err) return set_error(DLO_ERR_INVALID_ARG, "attention: null pointer");
    if (R <= 0 || T <= 0 || H <= 0) return set_error(DLO_ERR_INVALID_ARG, "attention: non-positive size");
    if (H > 65535 || R > 65535) return set_error(DLO_ERR_SHAPE, "attention: too many heads or requests");
    if (reinterpret_cast<uintptr_t>(qkv) % 16 || reinterpret_cast<uintptr_t>(o) % 16)
        return set_error(DLO_ERR_ALIGNMENT, "attention: qkv and o must be 16-byte aligned");
    if (d == 64) return launch_attention_t<64>(qkv, R, T, H, o, err, st);
    if (d == 128) return launch_attention_t<128>(qkv, R, T, H, o, err, st);
    return set_error(DLO_ERR_SHAPE, "attention: head dim %d not supported (64 or 128)", d);
}

}  // namespace dlo
