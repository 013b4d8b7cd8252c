// Causal attention on the 5th-generation tensor cores, head dim 128, bf16.
//
// Source: nanochat speedrun walkthrough (lyylswood.com), section 预搜检
// (pretraining): 10 heads of dim 128 at d20, causal next-token model.
//   forward:  O_t = sum_{s<=t} softmax_s(q_t.k_s / sqrt(D)) v_s, with the
//             natural-log sum-exp lse_t kept for the backward;
//   backward: P = exp(S - lse), dP = dO V^T, D_t = dO_t.O_t,
//             dS = P (dP - D); dq = dS K / sqrt(D), dk = dS^T Q / sqrt(D),
//             dv = P^T dO.
//
// Every tile is 128 rows x 128 head-dim columns of bf16 held in shared
// memory as two 128-byte-swizzled atoms of 64 columns (the TMA layout).  The
// same bytes serve as a K-major operand (K = the 128 columns) and as an
// MN-major operand (K = the 128 rows), so K, V, Q and dO are loaded once and
// used in both orientations.  One CTA: warp 0 issues TMA loads, warp 1
// issues tcgen05.mma from one thread, warps 2-5 (128 threads, one row each)
// do the softmax arithmetic on rows read from TMEM and write bf16 operand
// tiles back to shared memory.
//
// forward (one CTA per 128-query block, keys in 128-blocks up to the diagonal):
//   S_j = Q K_j^T into one of two TMEM buffers (the next S overlaps the
//   softmax of this one); P_j = exp2(S_j*c - m) to shared memory; O += P_j V_j
//   in TMEM.  The running max m is raised only when it grows by more than
//   2^8, and O is then rescaled in TMEM (the rescale is rare after the first
//   blocks; P stays <= 256).
// backward, deterministic, no atomics:
//   dK/dV kernel, one CTA per 128-key block, query blocks from the diagonal on:
//     S^T = K Q^T, dP^T = V dO^T, P^T and dS^T through one shared tile,
//     dV += P^T dO, dK += dS^T Q accumulated in TMEM;
//   dQ kernel, one CTA per 128-query block, key blocks up to the diagonal:
//     S = Q K^T, dP = dO V^T, dS to shared memory, dQ += dS K in TMEM.
#include "kernels.cuh"
#include "tc_ptx.cuh"

namespace nc {
namespace {

constexpr int HD = 128;                 // head dim of this path
constexpr int BR = 128;                 // rows per block
constexpr int ATOM = BR * 64 * 2;       // 16 KB: 128 rows x 64 bf16, 128-byte swizzle
constexpr int TILE = 2 * ATOM;          // 32 KB
constexpr int NT = 192;
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;
constexpr uint32_t IDESC_KK = tc::idesc_bf16(128, 128, false, false);
constexpr uint32_t IDESC_KM = tc::idesc_bf16(128, 128, false, true);

// K-major view of a tile (K = its 128 columns), k-th 16-column slice.
__device__ __forceinline__ uint64_t dk_(uint32_t tile, int kk) {
    return tc::sdesc(tile + (kk >> 2) * ATOM + (kk & 3) * 32, 16, 1024);
}
// MN-major view of a tile (MN = its columns, K = its rows), k-th 16-row slice.
__device__ __forceinline__ uint64_t dm_(uint32_t tile, int kk) {
    return tc::sdesc(tile + kk * 2048, ATOM, 1024);
}

__device__ __forceinline__ void load_tile(uint8_t* dst, const CUtensorMap* m, uint64_t* bar, int col0,
                                          int row0) {
    tc::tma_load_3d(dst, m, bar, col0, row0, 0);
    tc::tma_load_3d(dst + ATOM, m, bar, col0 + 64, row0, 0);
}

__device__ __forceinline__ uint32_t pack2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

// Row r of a tile from 64 packed bf16 pairs, in the 128-byte swizzle.
__device__ __forceinline__ void store_row(uint8_t* tile, int r, const uint32_t* w) {
#pragma unroll
    for (int c = 0; c < 16; ++c) {
        uint8_t* dst = tile + (c >> 3) * ATOM + r * 128 + (((c & 7) ^ (r & 7)) << 4);
        *reinterpret_cast<uint4*>(dst) = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
    }
}

__device__ __forceinline__ void ld_row128(uint32_t taddr, float* v) {
#pragma unroll
    for (int c = 0; c < 4; ++c) tc::tmem_ld32(taddr + c * 32, reinterpret_cast<uint32_t*>(v) + c * 32);
    tc::tmem_wait_ld();
}

__device__ __forceinline__ void store_out_row(bf16* dst, const float* v, float scale) {
#pragma unroll
    for (int c = 0; c < 16; ++c) {
        uint4 u = make_uint4(pack2(v[8 * c] * scale, v[8 * c + 1] * scale), pack2(v[8 * c + 2] * scale, v[8 * c + 3] * scale),
                             pack2(v[8 * c + 4] * scale, v[8 * c + 5] * scale), pack2(v[8 * c + 6] * scale, v[8 * c + 7] * scale));
        reinterpret_cast<uint4*>(dst)[c] = u;
    }
}

struct AttnParams {
    int T, H, nblk;        // sequence length, heads, 128-blocks per sequence
    long ldo;              // row stride of O / dO (forward out, backward in)
    long ldd;              // row stride of dq/dk/dv
    bf16* o;               // forward output
    float* lse;            // [B, H, T]
    const float* delta;    // [B, H, T] (backward)
    bf16 *dq, *dk, *dv;    // backward outputs
    float scale;           // 1/sqrt(D)
    uint32_t* flag;
};

struct Smem {
    uint8_t* base;
    uint64_t* bar;
    uint32_t* tmem_slot;
    volatile int* abort;
};

__device__ __forceinline__ Smem carve(uint8_t* raw, int ntiles) {
    Smem s;
    s.base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~(uintptr_t)1023);
    s.bar = reinterpret_cast<uint64_t*>(s.base + ntiles * TILE);
    s.tmem_slot = reinterpret_cast<uint32_t*>(s.bar + 24);
    s.abort = reinterpret_cast<volatile int*>(s.tmem_slot + 1);
    return s;
}

__device__ __forceinline__ void setup(Smem& s, int nbar, const uint32_t* counts) {
    if (threadIdx.x == 0) {
        for (int i = 0; i < nbar; ++i) tc::mbar_init(&s.bar[i], counts[i]);
        *s.abort = 0;
        tc::fence_barrier_init();
    }
    if (threadIdx.x / 32 == 1) {
        tc::tmem_alloc(s.tmem_slot, 512);
        tc::tmem_relinquish();
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
}

__device__ __forceinline__ void teardown(Smem& s, uint32_t tmem, uint32_t* flag) {
    tc::fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && *s.abort && flag) atomicOr(flag, NC_FLAG_TIMEOUT);
    if (threadIdx.x / 32 == 1) {
        tc::fence_after();
        tc::tmem_dealloc(tmem, 512);
    }
}

// ===================================================================== forward
// smem tiles: 0 Q | 1,2 K/V stage 0 | 3,4 K/V stage 1 | 5,6 P buffers
// barriers: 0 q_full, 1-2 kv_full, 3-4 kv_empty, 5-6 s_full, 7-8 p_full, 9-10 o_done
// TMEM: S buffers at columns 0 and 128, O at 256.
constexpr int FWD_TILES = 7;

__global__ void __launch_bounds__(NT, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                    const __grid_constant__ CUtensorMap mv, const AttnParams p) {
    extern __shared__ uint8_t smem_raw[];
    Smem sm = carve(smem_raw, FWD_TILES);
    const int qb = p.nblk - 1 - blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int nkb = qb + 1;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    uint64_t* q_full = &sm.bar[0];
    uint64_t* kv_full = &sm.bar[1];
    uint64_t* kv_empty = &sm.bar[3];
    uint64_t* s_full = &sm.bar[5];
    uint64_t* p_full = &sm.bar[7];
    uint64_t* o_done = &sm.bar[9];
    const uint32_t counts[11] = {1, 1, 1, 1, 1, 1, 1, 128, 128, 1, 1};
    setup(sm, 11, counts);
    const uint32_t tmem = *sm.tmem_slot;
    uint8_t* Q = sm.base;
    auto Kt = [&](int st) { return sm.base + (1 + 2 * st) * TILE; };
    auto Vt = [&](int st) { return sm.base + (2 + 2 * st) * TILE; };
    auto Pt = [&](int i) { return sm.base + (5 + i) * TILE; };
    const int col = h * HD;
    const int rowq = b * p.T + qb * BR;

    if (warp == 0 && lane == 0) {
        tc::mbar_expect_tx(q_full, TILE);
        load_tile(Q, &mq, q_full, col, rowq);
        for (int j = 0; j < nkb; ++j) {
            const int st = j & 1;
            if (!tc::mbar_wait(&kv_empty[st], ((j >> 1) & 1) ^ 1, sm.abort)) break;
            tc::mbar_expect_tx(&kv_full[st], 2 * TILE);
            load_tile(Kt(st), &mk, &kv_full[st], col, b * p.T + j * BR);
            load_tile(Vt(st), &mv, &kv_full[st], col, b * p.T + j * BR);
        }
    } else if (warp == 1 && lane == 0) {
        const uint32_t q0 = tc::smem_u32(Q);
        bool ok = tc::mbar_wait(q_full, 0, sm.abort);
        auto issue_s = [&](int j) -> bool {
            const int st = j & 1;
            if (!tc::mbar_wait(&kv_full[st], (j >> 1) & 1, sm.abort)) return false;
            tc::fence_after();
            const uint32_t k0 = tc::smem_u32(Kt(st));
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                tc::mma_bf16(tmem + (j & 1) * 128, dk_(q0, kk), dk_(k0, kk), IDESC_KK, kk > 0);
            tc::mma_commit(&s_full[j & 1]);
            return true;
        };
        if (ok) ok = issue_s(0);
        for (int j = 0; ok && j < nkb; ++j) {
            if (j + 1 < nkb && !issue_s(j + 1)) break;
            if (!tc::mbar_wait(&p_full[j & 1], (j >> 1) & 1, sm.abort)) break;
            tc::fence_after();
            const uint32_t p0 = tc::smem_u32(Pt(j & 1)), v0 = tc::smem_u32(Vt(j & 1));
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                tc::mma_bf16(tmem + 256, dk_(p0, kk), dm_(v0, kk), IDESC_KM, (j > 0 || kk > 0));
            tc::mma_commit(&o_done[j & 1]);
            tc::mma_commit(&kv_empty[j & 1]);
        }
    } else if (warp >= 2) {
        const int q = warp & 3, r = q * 32 + lane;
        const uint32_t lanes = (uint32_t)(q * 32) << 16;
        const float c2 = p.scale * LOG2E;
        float m2 = -INFINITY, l = 0.f;
        float s[128];
        bool ok = true;
        for (int j = 0; j < nkb; ++j) {
            if (!(ok = tc::mbar_wait_warp(&s_full[j & 1], (j >> 1) & 1, sm.abort))) break;
            tc::fence_after();
            ld_row128(tmem + lanes + (j & 1) * 128, s);
            float mx = -INFINITY;
            if (j == qb) {
#pragma unroll
                for (int i = 0; i < 128; ++i) {
                    s[i] = i > r ? -INFINITY : s[i] * c2;
                    mx = fmaxf(mx, s[i]);
                }
            } else {
#pragma unroll
                for (int i = 0; i < 128; ++i) {
                    s[i] *= c2;
                    mx = fmaxf(mx, s[i]);
                }
            }
            if (j == 0) {
                m2 = mx;
            } else {
                const bool need = mx > m2 + 8.f;
                if (__any_sync(0xffffffffu, need)) {
                    // O += P_{j-1} V_{j-1} must be complete before O is rescaled
                    if (!(ok = tc::mbar_wait_warp(&o_done[(j - 1) & 1], ((j - 1) >> 1) & 1, sm.abort))) break;
                    tc::fence_after();
                    const float alpha = need ? exp2f(m2 - mx) : 1.f;
#pragma unroll 1
                    for (int c = 0; c < 4; ++c) {
                        uint32_t o[32];
                        tc::tmem_ld32(tmem + lanes + 256 + c * 32, o);
                        tc::tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                        tc::tmem_st32(tmem + lanes + 256 + c * 32, o);
                    }
                    tc::tmem_wait_st();
                    if (need) {
                        l *= alpha;
                        m2 = mx;
                    }
                }
            }
            uint32_t w[64];
            float sum = 0.f;
#pragma unroll
            for (int i = 0; i < 64; ++i) {
                const float a = exp2f(s[2 * i] - m2), bb = exp2f(s[2 * i + 1] - m2);
                sum += a + bb;
                w[i] = pack2(a, bb);
            }
            l += sum;
            if (j >= 2 && !(ok = tc::mbar_wait_warp(&o_done[j & 1], ((j - 2) >> 1) & 1, sm.abort))) break;
            store_row(Pt(j & 1), r, w);
            tc::fence_async_smem();
            tc::fence_before();
            tc::mbar_arrive(&p_full[j & 1]);
        }
        if (ok && tc::mbar_wait_warp(&o_done[(nkb - 1) & 1], ((nkb - 1) >> 1) & 1, sm.abort)) {
            tc::fence_after();
            ld_row128(tmem + lanes + 256, s);
            const int t = qb * BR + r;
            if (t < p.T) {
                store_out_row(p.o + (long)(b * p.T + t) * p.ldo + col, s, 1.f / l);
                p.lse[((long)b * p.H + h) * p.T + t] = (m2 + log2f(l)) * LN2;
            }
        }
    }
    teardown(sm, tmem, p.flag);
}

// ===================================================================== dQ
// smem tiles: 0 Q | 1 dO | 2,3 K/V stage 0 | 4,5 K/V stage 1 | 6 dS
// barriers: 0 qd_full, 1-2 kv_full, 3-4 kv_empty, 5 s_full, 6 s_free, 7 ds_full, 8 dq_done
// TMEM: S at 0, dP at 128, dQ at 256.
constexpr int DQ_TILES = 7;

__global__ void __launch_bounds__(NT, 1)
    attn_dq_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                   const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mdo,
                   const AttnParams p) {
    extern __shared__ uint8_t smem_raw[];
    Smem sm = carve(smem_raw, DQ_TILES);
    const int qb = p.nblk - 1 - blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int nkb = qb + 1;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    uint64_t* qd_full = &sm.bar[0];
    uint64_t* kv_full = &sm.bar[1];
    uint64_t* kv_empty = &sm.bar[3];
    uint64_t* s_full = &sm.bar[5];
    uint64_t* s_free = &sm.bar[6];
    uint64_t* ds_full = &sm.bar[7];
    uint64_t* dq_done = &sm.bar[8];
    const uint32_t counts[9] = {1, 1, 1, 1, 1, 1, 128, 128, 1};
    setup(sm, 9, counts);
    const uint32_t tmem = *sm.tmem_slot;
    uint8_t* Q = sm.base;
    uint8_t* dO = sm.base + TILE;
    auto Kt = [&](int st) { return sm.base + (2 + 2 * st) * TILE; };
    auto Vt = [&](int st) { return sm.base + (3 + 2 * st) * TILE; };
    uint8_t* dS = sm.base + 6 * TILE;
    const int col = h * HD;
    const int rowq = b * p.T + qb * BR;

    if (warp == 0 && lane == 0) {
        tc::mbar_expect_tx(qd_full, 2 * TILE);
        load_tile(Q, &mq, qd_full, col, rowq);
        load_tile(dO, &mdo, qd_full, col, rowq);
        for (int j = 0; j < nkb; ++j) {
            const int st = j & 1;
            if (!tc::mbar_wait(&kv_empty[st], ((j >> 1) & 1) ^ 1, sm.abort)) break;
            tc::mbar_expect_tx(&kv_full[st], 2 * TILE);
            load_tile(Kt(st), &mk, &kv_full[st], col, b * p.T + j * BR);
            load_tile(Vt(st), &mv, &kv_full[st], col, b * p.T + j * BR);
        }
    } else if (warp == 1 && lane == 0) {
        const uint32_t q0 = tc::smem_u32(Q), do0 = tc::smem_u32(dO), ds0 = tc::smem_u32(dS);
        bool ok = tc::mbar_wait(qd_full, 0, sm.abort);
        for (int j = 0; ok && j < nkb; ++j) {
            const int st = j & 1;
            if (!(ok = tc::mbar_wait(&kv_full[st], (j >> 1) & 1, sm.abort))) break;
            // S and dP of the previous block must have been read out of TMEM
            if (j > 0 && !(ok = tc::mbar_wait(s_free, (j - 1) & 1, sm.abort))) break;
            tc::fence_after();
            const uint32_t k0 = tc::smem_u32(Kt(st)), v0 = tc::smem_u32(Vt(st));
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) tc::mma_bf16(tmem, dk_(q0, kk), dk_(k0, kk), IDESC_KK, kk > 0);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) tc::mma_bf16(tmem + 128, dk_(do0, kk), dk_(v0, kk), IDESC_KK, kk > 0);
            tc::mma_commit(s_full);
            if (!(ok = tc::mbar_wait(ds_full, j & 1, sm.abort))) break;
            tc::fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                tc::mma_bf16(tmem + 256, dk_(ds0, kk), dm_(k0, kk), IDESC_KM, (j > 0 || kk > 0));
            tc::mma_commit(dq_done);
            tc::mma_commit(&kv_empty[st]);
        }
    } else if (warp >= 2) {
        const int q = warp & 3, r = q * 32 + lane;
        const uint32_t lanes = (uint32_t)(q * 32) << 16;
        const float c2 = p.scale * LOG2E;
        const int t = qb * BR + r;
        const long st_i = ((long)b * p.H + h) * p.T + (t < p.T ? t : 0);
        const float lse2 = t < p.T ? p.lse[st_i] * LOG2E : INFINITY;
        const float Dt = t < p.T ? p.delta[st_i] : 0.f;
        float s[128];
        bool ok = true;
        for (int j = 0; j < nkb; ++j) {
            if (!(ok = tc::mbar_wait_warp(s_full, j & 1, sm.abort))) break;
            tc::fence_after();
            ld_row128(tmem + lanes, s);
#pragma unroll
            for (int i = 0; i < 128; ++i) s[i] = (j == qb && i > r) ? 0.f : exp2f(s[i] * c2 - lse2);
            uint32_t w[64];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t d[32];
                tc::tmem_ld32(tmem + lanes + 128 + c * 32, d);
                tc::tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    w[16 * c + i] = pack2(s[32 * c + 2 * i] * (__uint_as_float(d[2 * i]) - Dt),
                                          s[32 * c + 2 * i + 1] * (__uint_as_float(d[2 * i + 1]) - Dt));
            }
            tc::fence_before();
            tc::mbar_arrive(s_free);
            // the previous dQ MMA must be done reading the dS tile
            if (j > 0 && !(ok = tc::mbar_wait_warp(dq_done, (j - 1) & 1, sm.abort))) break;
            store_row(dS, r, w);
            tc::fence_async_smem();
            tc::fence_before();
            tc::mbar_arrive(ds_full);
        }
        if (ok && tc::mbar_wait_warp(dq_done, (nkb - 1) & 1, sm.abort)) {
            tc::fence_after();
            ld_row128(tmem + lanes + 256, s);
            if (t < p.T) store_out_row(p.dq + (long)(b * p.T + t) * p.ldd + col, s, p.scale);
        }
    }
    teardown(sm, tmem, p.flag);
}

// ===================================================================== dK, dV
// smem tiles: 0 K | 1 V | 2,3 Q/dO stage 0 | 4,5 Q/dO stage 1 | 6 P^T then dS^T
// barriers: 0 kv_full, 1-2 qd_full, 3-4 qd_empty, 5 s_full, 6 s_free, 7 p_full, 8 dv_done,
//           9 ds_full, 10 dk_done
// TMEM: S^T at 0, dP^T at 128, dV at 256, dK at 384.
constexpr int DKV_TILES = 7;

__global__ void __launch_bounds__(NT, 1)
    attn_dkdv_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                     const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mdo,
                     const AttnParams p) {
    extern __shared__ uint8_t smem_raw[];
    Smem sm = carve(smem_raw, DKV_TILES);
    const int kb = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int nq = p.nblk - kb;        // query blocks kb .. nblk-1
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    uint64_t* kv_full = &sm.bar[0];
    uint64_t* qd_full = &sm.bar[1];
    uint64_t* qd_empty = &sm.bar[3];
    uint64_t* s_full = &sm.bar[5];
    uint64_t* s_free = &sm.bar[6];
    uint64_t* p_full = &sm.bar[7];
    uint64_t* dv_done = &sm.bar[8];
    uint64_t* ds_full = &sm.bar[9];
    uint64_t* dk_done = &sm.bar[10];
    const uint32_t counts[11] = {1, 1, 1, 1, 1, 1, 128, 128, 1, 128, 1};
    setup(sm, 11, counts);
    const uint32_t tmem = *sm.tmem_slot;
    uint8_t* K = sm.base;
    uint8_t* V = sm.base + TILE;
    auto Qt = [&](int st) { return sm.base + (2 + 2 * st) * TILE; };
    auto dOt = [&](int st) { return sm.base + (3 + 2 * st) * TILE; };
    uint8_t* PS = sm.base + 6 * TILE;
    const int col = h * HD;
    const int rowk = b * p.T + kb * BR;

    if (warp == 0 && lane == 0) {
        tc::mbar_expect_tx(kv_full, 2 * TILE);
        load_tile(K, &mk, kv_full, col, rowk);
        load_tile(V, &mv, kv_full, col, rowk);
        for (int i = 0; i < nq; ++i) {
            const int st = i & 1, j = kb + i;
            if (!tc::mbar_wait(&qd_empty[st], ((i >> 1) & 1) ^ 1, sm.abort)) break;
            tc::mbar_expect_tx(&qd_full[st], 2 * TILE);
            load_tile(Qt(st), &mq, &qd_full[st], col, b * p.T + j * BR);
            load_tile(dOt(st), &mdo, &qd_full[st], col, b * p.T + j * BR);
        }
    } else if (warp == 1 && lane == 0) {
        const uint32_t k0 = tc::smem_u32(K), v0 = tc::smem_u32(V), ps0 = tc::smem_u32(PS);
        bool ok = tc::mbar_wait(kv_full, 0, sm.abort);
        auto issue_s = [&](int i) -> bool {
            const int st = i & 1;
            if (!tc::mbar_wait(&qd_full[st], (i >> 1) & 1, sm.abort)) return false;
            if (i > 0 && !tc::mbar_wait(s_free, (i - 1) & 1, sm.abort)) return false;
            tc::fence_after();
            const uint32_t q0 = tc::smem_u32(Qt(st)), do0 = tc::smem_u32(dOt(st));
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) tc::mma_bf16(tmem, dk_(k0, kk), dk_(q0, kk), IDESC_KK, kk > 0);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) tc::mma_bf16(tmem + 128, dk_(v0, kk), dk_(do0, kk), IDESC_KK, kk > 0);
            tc::mma_commit(s_full);
            return true;
        };
        if (ok) ok = issue_s(0);
        for (int i = 0; ok && i < nq; ++i) {
            const int st = i & 1;
            const uint32_t q0 = tc::smem_u32(Qt(st)), do0 = tc::smem_u32(dOt(st));
            if (!(ok = tc::mbar_wait(p_full, i & 1, sm.abort))) break;
            tc::fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                tc::mma_bf16(tmem + 256, dk_(ps0, kk), dm_(do0, kk), IDESC_KM, (i > 0 || kk > 0));
            tc::mma_commit(dv_done);
            if (i + 1 < nq && !(ok = issue_s(i + 1))) break;
            if (!(ok = tc::mbar_wait(ds_full, i & 1, sm.abort))) break;
            tc::fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                tc::mma_bf16(tmem + 384, dk_(ps0, kk), dm_(q0, kk), IDESC_KM, (i > 0 || kk > 0));
            tc::mma_commit(dk_done);
            tc::mma_commit(&qd_empty[st]);
        }
    } else if (warp >= 2) {
        const int q = warp & 3, r = q * 32 + lane;   // r = key row within the block
        const uint32_t lanes = (uint32_t)(q * 32) << 16;
        const float c2 = p.scale * LOG2E;
        float s[128];
        bool ok = true;
        const long srow = ((long)b * p.H + h) * p.T;   // statistics of this (b, h)
        for (int i = 0; i < nq; ++i) {
            const int j = kb + i;
            const int tq = j * BR;                       // first query of the block
            const int nvalid = p.T - tq;                 // queries c >= nvalid are padding
            if (!(ok = tc::mbar_wait_warp(s_full, i & 1, sm.abort))) break;
            tc::fence_after();
            ld_row128(tmem + lanes, s);
            // P^T[r][c] = exp2(S^T*c2 - lse2[c]), zero where key r > query c
#pragma unroll
            for (int c = 0; c < 128; ++c) {
                // every thread reads the same statistic: one broadcast load per warp
                const float l2 = c < nvalid ? __ldg(p.lse + srow + tq + c) * LOG2E : INFINITY;
                s[c] = (i == 0 && r > c) ? 0.f : exp2f(s[c] * c2 - l2);
            }
            uint32_t w[64];
#pragma unroll
            for (int c = 0; c < 64; ++c) w[c] = pack2(s[2 * c], s[2 * c + 1]);
            if (i > 0 && !(ok = tc::mbar_wait_warp(dk_done, (i - 1) & 1, sm.abort))) break;
            store_row(PS, r, w);
            tc::fence_async_smem();
            tc::fence_before();
            tc::mbar_arrive(p_full);
            // dS^T = P^T (dP^T - D[c])
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t d[32];
                tc::tmem_ld32(tmem + lanes + 128 + c * 32, d);
                tc::tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int c0 = 32 * c + 2 * e;
                    const float d0 = c0 < nvalid ? __ldg(p.delta + srow + tq + c0) : 0.f;
                    const float d1 = c0 + 1 < nvalid ? __ldg(p.delta + srow + tq + c0 + 1) : 0.f;
                    w[16 * c + e] = pack2(s[c0] * (__uint_as_float(d[2 * e]) - d0),
                                          s[c0 + 1] * (__uint_as_float(d[2 * e + 1]) - d1));
                }
            }
            tc::fence_before();
            tc::mbar_arrive(s_free);
            if (!(ok = tc::mbar_wait_warp(dv_done, i & 1, sm.abort))) break;
            store_row(PS, r, w);
            tc::fence_async_smem();
            tc::fence_before();
            tc::mbar_arrive(ds_full);
        }
        if (ok && tc::mbar_wait_warp(dk_done, (nq - 1) & 1, sm.abort)) {
            tc::fence_after();
            const int key = kb * BR + r;
            ld_row128(tmem + lanes + 256, s);
            if (key < p.T) store_out_row(p.dv + (long)(b * p.T + key) * p.ldd + col, s, 1.f);
            ld_row128(tmem + lanes + 384, s);
            if (key < p.T) store_out_row(p.dk + (long)(b * p.T + key) * p.ldd + col, s, p.scale);
        }
    }
    teardown(sm, tmem, p.flag);
}

int smem_bytes(int tiles) { return tiles * TILE + 1024 + 256; }

template <typename K>
int set_smem(K kern, int bytes) {
    return cuda_check(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes),
                      "attention smem attribute");
}

int maps(CUtensorMap* m, const void* ptr, long rows, long ld, int H) {
    return make_map(m, ptr, (long)H * HD, rows, 1, ld, 0, 64, BR);
}

}  // namespace

uint32_t* g_attn_flag = nullptr;

bool attention_tc_supported(long ld, long ldo, long ldd, const void* q, const void* k, const void* v,
                            int D) {
    if (D != HD) return false;
    if (ld % 8 || ldo % 8 || ldd % 8) return false;
    if ((uintptr_t)q % 16 || (uintptr_t)k % 16 || (uintptr_t)v % 16) return false;
    return true;
}

int attention_forward_tc(const bf16* q, const bf16* k, const bf16* v, long ld, bf16* o, long ldo,
                         float* lse, int B, int T, int H, cudaStream_t s) {
    static bool init = false;
    if (!init) {
        NC_TRY(set_smem(attn_fwd_kernel, smem_bytes(FWD_TILES)));
        init = true;
    }
    CUtensorMap mq, mk, mv;
    const long rows = (long)B * T;
    NC_TRY(maps(&mq, q, rows, ld, H));
    NC_TRY(maps(&mk, k, rows, ld, H));
    NC_TRY(maps(&mv, v, rows, ld, H));
    AttnParams p{};
    p.T = T; p.H = H; p.nblk = ceil_div(T, BR); p.ldo = ldo; p.o = o; p.lse = lse;
    p.scale = 1.0f / sqrtf((float)HD); p.flag = g_attn_flag;
    attn_fwd_kernel<<<dim3(p.nblk, H, B), NT, smem_bytes(FWD_TILES), s>>>(mq, mk, mv, p);
    note_launch();
    NC_LAUNCH_CHECK("attn_fwd_kernel");
    return NC_OK;
}

int attention_backward_tc(const bf16* q, const bf16* k, const bf16* v, long ld, const bf16* dout,
                          long ldo, const float* lse, const float* delta, bf16* dq, bf16* dk, bf16* dv,
                          long ldd, int B, int T, int H, cudaStream_t s) {
    static bool init = false;
    if (!init) {
        NC_TRY(set_smem(attn_dq_kernel, smem_bytes(DQ_TILES)));
        NC_TRY(set_smem(attn_dkdv_kernel, smem_bytes(DKV_TILES)));
        init = true;
    }
    CUtensorMap mq, mk, mv, mdo;
    const long rows = (long)B * T;
    NC_TRY(maps(&mq, q, rows, ld, H));
    NC_TRY(maps(&mk, k, rows, ld, H));
    NC_TRY(maps(&mv, v, rows, ld, H));
    NC_TRY(maps(&mdo, dout, rows, ldo, H));
    AttnParams p{};
    p.T = T; p.H = H; p.nblk = ceil_div(T, BR); p.ldo = ldo; p.ldd = ldd;
    p.lse = const_cast<float*>(lse); p.delta = delta; p.dq = dq; p.dk = dk; p.dv = dv;
    p.scale = 1.0f / sqrtf((float)HD); p.flag = g_attn_flag;
    attn_dkdv_kernel<<<dim3(p.nblk, H, B), NT, smem_bytes(DKV_TILES), s>>>(mq, mk, mv, mdo, p);
    attn_dq_kernel<<<dim3(p.nblk, H, B), NT, smem_bytes(DQ_TILES), s>>>(mq, mk, mv, mdo, p);
    note_launch(2);
    NC_LAUNCH_CHECK("attn backward kernels");
    return NC_OK;
}

}  // namespace nc
