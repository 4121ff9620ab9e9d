// Non-causal multi-head softmax attention of the DiT block, one request at a
// time (requests never attend to each other).
//
// qkv bf16 [R*T, 3h]: q | k | v column groups, head j at columns j*d of each.
// o   bf16 [R*T, h] : head j at columns j*d.
// O = softmax(Q K^T / sqrt(d)) V, fp32 logits, fp32 online softmax
// (running max and sum, rescaled per key tile), fp32 accumulation.
//
// One CTA = 64 query rows of one (request, head); 4 warps x 16 rows.  Key /
// value tiles of 64 rows are double-buffered in shared memory with cp.async;
// rows past T are zero-filled and their logits masked to -inf.  Products use
// mma.sync m16n8k16 bf16 -> fp32 with ldmatrix fragments; the 16-byte chunks
// of every shared row are XOR-swizzled by (row % 8) to avoid bank conflicts.
#include "dlo_device.cuh"
#include "dlo_internal.h"

namespace dlo {

namespace {

constexpr int kAttBQ = 64;
constexpr int kAttBKV = 64;
constexpr int kAttThreads = 128;

__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, bool valid) {
    const int n = valid ? 16 : 0;  // 0 source bytes: the 16 destination bytes are zero-filled
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void mma_16816(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Byte offset of 16-byte chunk `ch` of row `row` in a [rows][D] bf16 tile.
template <int D>
__device__ __forceinline__ uint32_t swz(int row, int ch) {
    return (uint32_t)(row * (D * 2) + ((ch ^ (row & 7)) << 4));
}

// Loads `rows` rows (tile start t0) of one head's D columns into a swizzled tile.
template <int D>
__device__ __forceinline__ void load_tile(uint32_t s_base, const uint16_t* g, int ld, int t0, int T) {
    constexpr int CH = D / 8;
    for (int i = threadIdx.x; i < kAttBKV * CH; i += kAttThreads) {
        const int row = i / CH, ch = i % CH;
        const int t = t0 + row;
        const bool valid = t < T;
        const uint16_t* src = g + (size_t)(valid ? t : 0) * ld + ch * 8;
        cp_async_16(s_base + swz<D>(row, ch), src, valid);
    }
}

}  // namespace

template <int D>
__global__ void __launch_bounds__(kAttThreads) attention_fwd_mma(const uint16_t* __restrict__ qkv, int T, int H,
                                                                   uint16_t* __restrict__ o, float scale_log2) {
    constexpr int TILE = kAttBKV * D * 2;  // bytes of one 64-row tile
    extern __shared__ __align__(128) uint8_t smem[];
    const uint32_t sQ = smem_u32(smem);
    const uint32_t sK0 = sQ + TILE;          // K buffers at sK0 + b*TILE
    const uint32_t sV0 = sQ + 3 * TILE;      // V buffers at sV0 + b*TILE

    const int q0 = blockIdx.x * kAttBQ;
    const int head = blockIdx.y;
    const int req = blockIdx.z;
    const int h = H * D;
    const int ld = 3 * h;
    const uint16_t* base = qkv + (size_t)req * T * ld;
    const uint16_t* gq = base + head * D;
    const uint16_t* gk = base + h + head * D;
    const uint16_t* gv = base + 2 * h + head * D;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t4 = lane & 3;
    const int nkv = (T + kAttBKV - 1) / kAttBKV;

    load_tile<D>(sQ, gq, ld, q0, T);
    load_tile<D>(sK0, gk, ld, 0, T);
    load_tile<D>(sV0, gv, ld, 0, T);
    cp_async_commit();

    uint32_t qf[D / 16][4];
    float oacc[D / 8][4];
#pragma unroll
    for (int i = 0; i < D / 8; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY};
    float l_run[2] = {0.f, 0.f};

    for (int j = 0; j < nkv; ++j) {
        const int buf = j & 1;
        if (j + 1 < nkv) {
            load_tile<D>(sK0 + (buf ^ 1) * TILE, gk, ld, (j + 1) * kAttBKV, T);
            load_tile<D>(sV0 + (buf ^ 1) * TILE, gv, ld, (j + 1) * kAttBKV, T);
            cp_async_commit();
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();

        if (j == 0) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const int mi = lane >> 3;
                const int row = warp * 16 + (mi & 1) * 8 + (lane & 7);
                const int ch = 2 * kk + (mi >> 1);
                ldsm_x4(sQ + swz<D>(row, ch), qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3]);
            }
        }

        // S = Q K^T for this warp's 16 rows x 64 keys
        const uint32_t sK = sK0 + buf * TILE;
        float s[8][4];
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
            s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < D / 16; kk += 2) {
                uint32_t b0, b1, b2, b3;
                const int row = nt * 8 + (lane & 7);
                const int ch = 2 * kk + (lane >> 3);
                ldsm_x4(sK + swz<D>(row, ch), b0, b1, b2, b3);
                mma_16816(s[nt], qf[kk], b0, b1);
                mma_16816(s[nt], qf[kk + 1], b2, b3);
            }
        }

        // mask keys past T (only the last tile can have them)
        const int kbase = j * kAttBKV;
        if (kbase + kAttBKV > T) {
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
                const int c = kbase + nt * 8 + 2 * t4;
                if (c >= T) s[nt][0] = s[nt][2] = -INFINITY;
                if (c + 1 >= T) s[nt][1] = s[nt][3] = -INFINITY;
            }
        }

        // online softmax (rows g and g+8 of the warp's 16)
        float mx[2] = {m_run[0], m_run[1]};
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
            mx[0] = fmaxf(mx[0], fmaxf(s[nt][0], s[nt][1]));
            mx[1] = fmaxf(mx[1], fmaxf(s[nt][2], s[nt][3]));
        }
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
            mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
        }
        float alpha[2], msc[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            alpha[r] = exp2f((m_run[r] - mx[r]) * scale_log2);
            m_run[r] = mx[r];
            msc[r] = mx[r] * scale_log2;
        }
        float rs[2] = {0.f, 0.f};
        uint32_t pf[4][4];  // P as bf16 A fragments, one per 16-key step
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
            const float p0 = exp2f(fmaf(s[nt][0], scale_log2, -msc[0]));
            const float p1 = exp2f(fmaf(s[nt][1], scale_log2, -msc[0]));
            const float p2 = exp2f(fmaf(s[nt][2], scale_log2, -msc[1]));
            const float p3 = exp2f(fmaf(s[nt][3], scale_log2, -msc[1]));
            rs[0] += p0 + p1;
            rs[1] += p2 + p3;
            const int kk = nt >> 1;
            if ((nt & 1) == 0) {
                pf[kk][0] = pack_bf16x2(p0, p1);
                pf[kk][1] = pack_bf16x2(p2, p3);
            } else {
                pf[kk][2] = pack_bf16x2(p0, p1);
                pf[kk][3] = pack_bf16x2(p2, p3);
            }
        }
#pragma unroll
        for (int r = 0; r < 2; ++r) l_run[r] = l_run[r] * alpha[r] + rs[r];
#pragma unroll
        for (int dt = 0; dt < D / 8; ++dt) {
            oacc[dt][0] *= alpha[0];
            oacc[dt][1] *= alpha[0];
            oacc[dt][2] *= alpha[1];
            oacc[dt][3] *= alpha[1];
        }

        // O += P V
        const uint32_t sV = sV0 + buf * TILE;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
            for (int dt = 0; dt < D / 8; dt += 2) {
                uint32_t b0, b1, b2, b3;
                const int mi = lane >> 3;
                const int row = kk * 16 + (mi & 1) * 8 + (lane & 7);
                const int ch = dt + (mi >> 1);
                ldsm_x4_t(sV + swz<D>(row, ch), b0, b1, b2, b3);
                mma_16816(oacc[dt], pf[kk], b0, b1);
                mma_16816(oacc[dt + 1], pf[kk], b2, b3);
            }
        }
        __syncthreads();
    }

    // normalise and store
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 1);
        l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 2);
    }
    const float inv0 = 1.f / l_run[0], inv1 = 1.f / l_run[1];
    const int r0 = q0 + warp * 16 + g;
    const int r1 = r0 + 8;
    uint16_t* ob = o + (size_t)req * T * h + head * D;
#pragma unroll
    for (int dt = 0; dt < D / 8; ++dt) {
        const int col = dt * 8 + 2 * t4;
        if (r0 < T)
            *reinterpret_cast<uint32_t*>(ob + (size_t)r0 * h + col) = pack_bf16x2(oacc[dt][0] * inv0, oacc[dt][1] * inv0);
        if (r1 < T)
            *reinterpret_cast<uint32_t*>(ob + (size_t)r1 * h + col) = pack_bf16x2(oacc[dt][2] * inv1, oacc[dt][3] * inv1);
    }
}

template <int D>
static int launch_attention_t(const uint16_t* qkv, int R, int T, int H, uint16_t* o, cudaStream_t st) {
    constexpr int smem = 5 * kAttBKV * D * 2;  // Q + 2 K + 2 V tiles
    static bool configured[64] = {};
    int dev = 0;
    DLO_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64) return set_error(DLO_ERR_INVALID_ARG, "device index %d out of range", dev);
    if (!configured[dev]) {
        DLO_CUDA_TRY(cudaFuncSetAttribute(attention_fwd_mma<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
        configured[dev] = true;
    }
    const float scale_log2 = 1.4426950408889634f / sqrtf((float)D);
    dim3 grid((T + kAttBQ - 1) / kAttBQ, H, R);
    attention_fwd_mma<D><<<grid, kAttThreads, smem, st>>>(qkv, T, H, o, scale_log2);
    DLO_CUDA_TRY(cudaGetLastError());
    return DLO_OK;
}

int launch_attention(const uint16_t* qkv, int R, int T, int H, int d, uint16_t* o, cudaStream_t st) {
    if (!qkv || !o) return set_error(DLO_ERR_INVALID_ARG, "attention: null pointer");
    if (R <= 0 || T <= 0 || H <= 0) return set_error(DLO_ERR_INVALID_ARG, "attention: non-positive size");
    if (H > 65535 || R > 65535) return set_error(DLO_ERR_SHAPE, "attention: too many heads or requests");
    if (d == 64) return launch_attention_t<64>(qkv, R, T, H, o, st);
    if (d == 128) return launch_attention_t<128>(qkv, R, T, H, o, st);
    return set_error(DLO_ERR_SHAPE, "attention: head dim %d not supported (64 or 128)", d);
}

}  // namespace dlo
