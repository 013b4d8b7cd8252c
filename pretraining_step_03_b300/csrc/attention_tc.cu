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
// issues tcgen05.mma from one thread, warps 2-9 do the softmax arithmetic on
// rows read from TMEM.  The probabilities (P, P^T) and score gradients (dS,
// dS^T) never touch shared memory: they are written back into TMEM as packed
// bf16 over the scores they came from and used from there as the A operand
// of the next product, which keeps shared-memory bandwidth for the operands
// TMA brings in (an M=128, N=128 MMA from shared memory already reads at the
// SM's shared-memory bandwidth).
//
// forward (one CTA per pair of 128-query blocks, keys in 128-blocks up to the diagonal):
//   S = Q K^T per query tile in TMEM; P = exp2(S*c - m) packed into TMEM over the
//   first half of its S; O += P V in TMEM.  One thread per query row; the two
//   tiles alternate on the tensor pipe (one tile's softmax overlaps the other
//   tile's products).  The running max m is raised only when it grows by more
//   than 2^8, and O is then rescaled in TMEM (rare after the first blocks; P
//   stays <= 256).  When given the RoPE table, the backward rotates dq and dk
//   back to the unrotated q, k frame in its epilogue.
// backward, deterministic, no atomics:
//   dK/dV kernel, one CTA per 128-key block, query blocks from the diagonal on:
//     S^T = K Q^T, dP^T = V dO^T, P^T and dS^T packed into TMEM,
//     dV += P^T dO, dK += dS^T Q accumulated in TMEM; given a dS store it also
//     writes each dS^T block (bf16) to global memory;
//   dQ, with the dS store: one CTA per 128-query block streams the stored dS
//     blocks and the K blocks up to the diagonal, dQ += dS K in TMEM (no
//     score is recomputed; the sum runs in key order, so it is deterministic);
//   dQ, without it: one CTA per 128-query block recomputes S = Q K^T and
//     dP = dO V^T, forms dS in TMEM and accumulates dQ += dS K.
#include "kernels.cuh"
#include "tc_ptx.cuh"

namespace nc {
namespace {

constexpr int HD = 128;                 // head dim of this path
constexpr int BR = 128;                 // rows per block
constexpr int ATOM = BR * 64 * 2;       // 16 KB: 128 rows x 64 bf16, 128-byte swizzle
constexpr int TILE = 2 * ATOM;          // 32 KB
constexpr int NT = 320;                 // producer warp, MMA warp, 8 softmax warps
constexpr int NSM = 256;                // softmax threads: 2 groups x 128 rows
constexpr int XCH_BYTES = 2048;         // [2 parities][2 groups][128] fp32 exchange / statistics
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

// A softmax thread of group g owns row r and the 32-column chunks g and g+2
// of a 128-column tile: columns [32g, 32g+32) and [64+32g, 64+32g+32), so a
// RoPE pair (j, j+64) of a head-dim row stays in one thread.
__device__ __forceinline__ int col_of(int g, int i) { return i < 32 ? 32 * g + i : 64 + 32 * g + (i - 32); }

__device__ __forceinline__ void ld_half(uint32_t taddr, int g, float* v) {
    tc::tmem_ld32(taddr + g * 32, reinterpret_cast<uint32_t*>(v));
    tc::tmem_ld32(taddr + (g + 2) * 32, reinterpret_cast<uint32_t*>(v) + 32);
    tc::tmem_wait_ld();
}

// this thread's 64 columns of an output row (bf16, row pointer at column 0)
__device__ __forceinline__ void store_out_half(bf16* row, int g, const float* v, float scale) {
#pragma unroll
    for (int a = 0; a < 2; ++a) {
        uint4* dst = reinterpret_cast<uint4*>(row + 64 * a + 32 * g);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float* x = v + 32 * a + 8 * k;
            dst[k] = make_uint4(pack2(x[0] * scale, x[1] * scale), pack2(x[2] * scale, x[3] * scale),
                                pack2(x[4] * scale, x[5] * scale), pack2(x[6] * scale, x[7] * scale));
        }
    }
}

// inverse RoPE (rotation by -angle) of head-dim pairs (j, j+64), j in [32g, 32g+32);
// the table is pair-major (pair j of position t at table[j * ld + t]), so the 32
// lanes of a warp (consecutive positions) read 256 contiguous bytes
__device__ __forceinline__ void unrope_half(float* v, const float2* table, int ld, int t, int g) {
    const float2* col = table + (long)(32 * g) * ld + t;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const float2 cs = __ldg(col + (long)i * ld);
        const float x1 = v[i], x2 = v[32 + i];
        v[i] = x1 * cs.x + x2 * cs.y;
        v[32 + i] = x2 * cs.x - x1 * cs.y;
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
    const float2* rope;    // (cos, sin) of pair j, position t at rope[j * rope_ld + t]; non-null:
    int rope_ld;           //   dq, dk leave rotated back
    bf16* ds;              // backward: dS tiles written by the dK/dV kernel (null: not kept)
    long ds_bh;            // tiles per (batch, head): nblk (nblk + 1) / 2
    float scale;           // 1/sqrt(D)
    uint32_t* flag;
};

// The dS store.  Tile (bh, i, j) holds dS of query block i, key block j <= i of
// batch-head bh; the tiles of one query block are consecutive (j = 0 .. i).  A
// tile is 32 KB: two 64-key halves of 16 KB, each [query/8][key%64][query%8]
// bf16, i.e. 16-byte chunks of 8 queries with the key fastest.  That order lets
// a warp (32 consecutive keys) write 512 contiguous bytes, and a half is the
// interleaved MN-major image of dS (M = queries, K = keys) that the dQ product
// copies to shared memory unchanged.
constexpr int DS_TILE = BR * HD * 2;
constexpr int DS_HALF = DS_TILE / 2;
__device__ __forceinline__ uint8_t* ds_tile(const AttnParams& p, int bh, int i, int j) {
    return reinterpret_cast<uint8_t*>(p.ds) + ((long)bh * p.ds_bh + (long)i * (i + 1) / 2 + j) * DS_TILE;
}

struct Smem {
    uint8_t* base;
    uint64_t* bar;
    uint32_t* tmem_slot;
    volatile int* abort;
    float* xch;            // [2][2][128]
};

__device__ __forceinline__ Smem carve(uint8_t* raw, int ntiles) {
    Smem s;
    s.base = raw;
    s.bar = reinterpret_cast<uint64_t*>(raw + ntiles * TILE);
    s.tmem_slot = reinterpret_cast<uint32_t*>(s.bar + 24);
    s.abort = reinterpret_cast<volatile int*>(s.tmem_slot + 1);
    s.xch = reinterpret_cast<float*>(raw + ntiles * TILE + 256);
    return s;
}

// The swizzled tiles need a 1024-byte aligned base; the launch asks for no
// slack, so a misaligned base is reported and the CTA does nothing.
__device__ __forceinline__ bool misaligned(const uint8_t* raw, uint32_t* flag) {
    if ((tc::smem_u32(raw) & 1023u) == 0) return false;
    if (threadIdx.x == 0 && flag) atomicOr(flag, NC_FLAG_SMEM_ALIGN);
    return true;
}

__device__ __forceinline__ void setup(Smem& s, int nbar, const uint32_t* counts, uint32_t ncols = 512) {
    if (threadIdx.x == 0) {
        for (int i = 0; i < nbar; ++i) tc::mbar_init(&s.bar[i], counts[i]);
        *s.abort = 0;
        tc::fence_barrier_init();
    }
    if (threadIdx.x / 32 == 1) {
        tc::tmem_alloc(s.tmem_slot, ncols);
        tc::tmem_relinquish();
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
}

__device__ __forceinline__ void teardown(Smem& s, uint32_t tmem, uint32_t* flag, uint32_t ncols = 512) {
    tc::fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && *s.abort && flag) atomicOr(flag, NC_FLAG_TIMEOUT);
    if (threadIdx.x / 32 == 1) {
        tc::fence_after();
        tc::tmem_dealloc(tmem, ncols);
    }
}


// write this thread's 64 probabilities, packed bf16 pairs, into row columns
// [16g, 16g+16) and [32+16g, 32+16g+16) of a TMEM region (the A-operand layout:
// word c holds keys 2c and 2c+1)
__device__ __forceinline__ void st_half_bf16(uint32_t taddr, int g, const uint32_t* w) {
    tc::tmem_st16(taddr + 16 * g, w);
    tc::tmem_st16(taddr + 32 + 16 * g, w + 16);
}

// ===================================================================== forward
// One CTA per pair of consecutive 128-query blocks (tiles 0 and 1) of one batch-head;
// both tiles stream the same K/V blocks.  Warps 2-5 do the softmax of tile 0 and
// warps 6-9 that of tile 1, one thread per query row holding its whole 128-key score
// row.  The MMA warp interleaves the tiles,
//   PV_0(j), S_0(j+1), PV_1(j), S_1(j+1), PV_0(j+1), ...
// so while one tile's softmax runs the tensor pipe works on the other tile.  S_t(j+1)
// overwrites the TMEM columns whose packed P_t(j) PV_t(j) reads, so it is issued once
// PV_t(j) has completed (an MMA's TMEM writes are not ordered after an earlier MMA's
// TMEM operand reads); that also keeps O_t still while the softmax rescales it.
// smem tiles: 0 Q_0 | 1 Q_1 | 2,3 K stages | 4,5 V stages
// barriers: 0 q_full, 1-2 k_full, 3-4 k_empty, 5-6 v_full, 7-8 v_empty, 9-10 s_full[t],
//           11-12 p_full[t], 13-14 o_done[t], 15 drain
// TMEM: S_t at 128 t (P_t packed into its first 64 columns), O_t at 256 + 128 t.
constexpr int FWD_TILES = 6;
constexpr int FWD_NST = 2;
constexpr int NSM_T = 128;   // softmax threads per tile

__global__ void __launch_bounds__(NT, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                    const __grid_constant__ CUtensorMap mv, const AttnParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    if (misaligned(smem_raw, p.flag)) return;
    Smem sm = carve(smem_raw, FWD_TILES);
    // the heaviest (latest) query-block pairs first; the pairs of one batch-head together
    const int npair = (p.nblk + 1) / 2;
    const int bh = blockIdx.y, c = npair - 1 - (int)blockIdx.x, h = bh % p.H, b = bh / p.H;
    if (c < 0) return;                 // (a grid wider than the sequence: nothing to do)
    const int qb0 = 2 * c;
    const bool has1 = qb0 + 1 < p.nblk;
    const int nk = has1 ? qb0 + 2 : qb0 + 1;          // key blocks streamed (tile t uses 0 .. qb0 + t)
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    uint64_t* q_full = &sm.bar[0];
    uint64_t* k_full = &sm.bar[1];
    uint64_t* k_empty = &sm.bar[3];
    uint64_t* v_full = &sm.bar[5];
    uint64_t* v_empty = &sm.bar[7];
    uint64_t* s_full = &sm.bar[9];
    uint64_t* p_full = &sm.bar[11];
    uint64_t* o_done = &sm.bar[13];
    uint64_t* drain = &sm.bar[15];
    const uint32_t counts[16] = {1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1, NSM_T, NSM_T, 1, 1, 1};
    setup(sm, 16, counts);
    const uint32_t tmem = *sm.tmem_slot;
    auto Qt = [&](int t) { return sm.base + t * TILE; };
    auto Kt = [&](int st) { return sm.base + (2 + st) * TILE; };
    auto Vt = [&](int st) { return sm.base + (2 + FWD_NST + st) * TILE; };
    const int col = h * HD;

    if (warp == 0 && lane == 0) {
        tc::mbar_expect_tx(q_full, (has1 ? 2 : 1) * TILE);
        load_tile(Qt(0), &mq, q_full, col, b * p.T + qb0 * BR);
        if (has1) load_tile(Qt(1), &mq, q_full, col, b * p.T + (qb0 + 1) * BR);
        int issued = 0;
        for (int j = 0; j < nk; ++j) {
            const int st = j % FWD_NST;
            const uint32_t ph = ((j / FWD_NST) & 1) ^ 1;
            if (!tc::mbar_wait(&k_empty[st], ph, sm.abort)) break;
            tc::mbar_expect_tx(&k_full[st], TILE);
            load_tile(Kt(st), &mk, &k_full[st], col, b * p.T + j * BR);
            if (!tc::mbar_wait(&v_empty[st], ph, sm.abort)) break;
            tc::mbar_expect_tx(&v_full[st], TILE);
            load_tile(Vt(st), &mv, &v_full[st], col, b * p.T + j * BR);
            issued = j + 1;
        }
        if (*sm.abort) {   // let the copies still in flight land before the CTA exits
            tc::mbar_wait_drain(q_full, 0);
            for (int j = issued - 1; j >= 0 && j >= issued - FWD_NST; --j) {
                tc::mbar_wait_drain(&k_full[j % FWD_NST], (j / FWD_NST) & 1);
                tc::mbar_wait_drain(&v_full[j % FWD_NST], (j / FWD_NST) & 1);
            }
        }
    } else if (warp == 1 && lane == 0) {
        bool ok = tc::mbar_wait(q_full, 0, sm.abort);
        // S_t(j) = Q_t K_j^T into TMEM 128 t
        auto issue_s = [&](int t, int j) -> bool {
            if (j > 0 && !tc::mbar_wait(&o_done[t], (j - 1) & 1, sm.abort)) return false;
            tc::fence_after();
            const uint32_t q0 = tc::smem_u32(Qt(t)), k0 = tc::smem_u32(Kt(j % FWD_NST));
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) tc::mma_bf16(tmem + 128 * t, dk_(q0, kk), dk_(k0, kk), IDESC_KK, kk > 0);
            tc::mma_commit(&s_full[t]);
            return true;
        };
        // O_t += P_t(j) V_j, P_t(j) packed in TMEM 128 t
        auto issue_pv = [&](int t, int j) -> bool {
            if (!tc::mbar_wait(&p_full[t], j & 1, sm.abort)) return false;
            tc::fence_after();
            const uint32_t v0 = tc::smem_u32(Vt(j % FWD_NST));
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                tc::mma_bf16_ts(tmem + 256 + 128 * t, tmem + 128 * t + kk * 8, dm_(v0, kk), IDESC_KM,
                                (j > 0 || kk > 0));
            tc::mma_commit(&o_done[t]);
            return true;
        };
        auto wait_k = [&](int j) { return tc::mbar_wait(&k_full[j % FWD_NST], (j / FWD_NST) & 1, sm.abort); };
        auto wait_v = [&](int j) { return tc::mbar_wait(&v_full[j % FWD_NST], (j / FWD_NST) & 1, sm.abort); };
        // tile 0 takes key blocks 0 .. nk0-1, tile 1 (if any) 0 .. nk-1
        const int nk0 = qb0 + 1;
        if (ok) ok = wait_k(0) && issue_s(0, 0) && (!has1 || issue_s(1, 0));
        if (ok) tc::mma_commit(&k_empty[0]);
        for (int j = 0; ok && j < nk; ++j) {
            if (!(ok = wait_v(j))) break;
            const bool next = j + 1 < nk;
            if (next && !(ok = wait_k(j + 1))) break;
            if (j < nk0) {
                if (!(ok = issue_pv(0, j))) break;
                if (j + 1 < nk0 && !(ok = issue_s(0, j + 1))) break;
            }
            if (has1) {
                if (!(ok = issue_pv(1, j))) break;
                if (next && !(ok = issue_s(1, j + 1))) break;
            }
            tc::mma_commit(&v_empty[j % FWD_NST]);
            if (next) tc::mma_commit(&k_empty[(j + 1) % FWD_NST]);
        }
        if (*sm.abort) {
            tc::mma_commit(drain);
            tc::mbar_wait_drain(drain, 0);
        }
    } else if (warp >= 2) {
        const int t = (warp - 2) >> 2, q = warp & 3, r = q * 32 + lane;
        const uint32_t lanes = (uint32_t)(q * 32) << 16;
        const int qb = qb0 + t;
        const int nkt = qb + 1;
        const float c2 = p.scale * LOG2E;
        float m2 = -INFINITY, l = 0.f;
        bool ok = t == 0 || has1;
        const uint32_t sb = tmem + lanes + 128 * t, ob = tmem + lanes + 256 + 128 * t;
        for (int j = 0; ok && j < nkt; ++j) {
            if (!(ok = tc::mbar_wait_warp(&s_full[t], j & 1, sm.abort))) break;
            tc::fence_after();
            float s[128];
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) tc::tmem_ld32(sb + 32 * cc, reinterpret_cast<uint32_t*>(s) + 32 * cc);
            tc::tmem_wait_ld();
            if (j == qb) {   // diagonal block: keys after the query are masked
#pragma unroll
                for (int i = 0; i < 128; ++i)
                    if (i > r) s[i] = -INFINITY;
            }
            float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int i = 0; i < 128; i += 2) m4[(i >> 1) & 3] = tc::fmax3(m4[(i >> 1) & 3], s[i], s[i + 1]);
            const float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * c2;   // log2 units
            // the running max moves only when it grows by more than 2^8 (P stays <= 256)
            const bool need = j > 0 && mx > m2 + 8.f;
            float alpha = 1.f;
            if (j == 0) m2 = mx;
            else if (need) {
                alpha = exp2f(m2 - mx);
                l *= alpha;
                m2 = mx;
            }
            // P_t(j) packed into the first 64 columns of S_t; scale, shift and the row sum
            // two lanes at a time
            const uint64_t c22 = tc::f2pk(c2, c2), nm2 = tc::f2pk(-m2, -m2);
            uint64_t sum2[2] = {tc::f2pk(0.f, 0.f), tc::f2pk(0.f, 0.f)};
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                uint32_t w[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    float a, bb;
                    tc::f2upk(tc::ffma2(tc::f2pk(s[64 * h2 + 2 * i], s[64 * h2 + 2 * i + 1]), c22, nm2), a, bb);
                    a = tc::ex2a(a);
                    bb = tc::ex2a(bb);
                    sum2[i & 1] = tc::fadd2(sum2[i & 1], tc::f2pk(a, bb));
                    w[i] = pack2(a, bb);
                }
                tc::tmem_st32(sb + 32 * h2, w);
            }
            {
                float x0, x1, y0, y1;
                tc::f2upk(sum2[0], x0, x1);
                tc::f2upk(sum2[1], y0, y1);
                l += (x0 + x1) + (y0 + y1);
            }
            if (__any_sync(0xffffffffu, need)) {
                // O_t is still (S_t(j) was issued after PV_t(j-1) completed): rescale in place
#pragma unroll 1
                for (int cc = 0; cc < 4; ++cc) {
                    uint32_t o[32];
                    tc::tmem_ld32(ob + 32 * cc, o);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                    tc::tmem_st32(ob + 32 * cc, o);
                }
            }
            tc::tmem_wait_st();
            tc::fence_before();
            tc::mbar_arrive(&p_full[t]);
        }
        if (ok && tc::mbar_wait_warp(&o_done[t], (nkt - 1) & 1, sm.abort)) {
            tc::fence_after();
            const int tq = qb * BR + r;
            const float inv = 1.f / l;
#pragma unroll 1
            for (int g = 0; g < 2; ++g) {
                float v[64];
                ld_half(ob, g, v);
                if (tq < p.T) store_out_half(p.o + (long)(b * p.T + tq) * p.ldo + col, g, v, inv);
            }
            if (tq < p.T) p.lse[((long)b * p.H + h) * p.T + tq] = (m2 + log2f(l)) * LN2;
        }
    }
    teardown(sm, tmem, p.flag);
}

// ===================================================================== dQ
// smem tiles: 0 Q | 1 dO | 2,3 K stages | 4,5 V stages
// barriers: 0 qd_full, 1-2 k_full, 3-4 k_empty, 5-6 v_full, 7-8 v_empty, 9 s_full, 10 ds_full,
//           11 dq_done
// TMEM: S at 0, dP at 128, dQ at 256, dS at 384 (packed bf16, the A operand of
// dQ += dS K).
constexpr int DQ_TILES = 6;

__global__ void __launch_bounds__(NT, 1)
    attn_dq_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                   const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mdo,
                   const AttnParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    if (misaligned(smem_raw, p.flag)) return;
    Smem sm = carve(smem_raw, DQ_TILES);
    const int bh = blockIdx.y, qb = p.nblk - 1 - (int)blockIdx.x, h = bh % p.H, b = bh / p.H;
    if (qb < 0) return;                // (a grid wider than the sequence: nothing to do)
    const int nkb = qb + 1;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    uint64_t* qd_full = &sm.bar[0];
    uint64_t* k_full = &sm.bar[1];
    uint64_t* k_empty = &sm.bar[3];
    uint64_t* v_full = &sm.bar[5];
    uint64_t* v_empty = &sm.bar[7];
    uint64_t* s_full = &sm.bar[9];
    uint64_t* ds_full = &sm.bar[10];
    uint64_t* dq_done = &sm.bar[11];
    const uint32_t counts[12] = {1, 1, 1, 1, 1, 1, 1, 1, 1, 1, NSM, 1};
    setup(sm, 12, counts);
    const uint32_t tmem = *sm.tmem_slot;
    uint8_t* Q = sm.base;
    uint8_t* dO = sm.base + TILE;
    auto Kt = [&](int st) { return sm.base + (2 + st) * TILE; };
    auto Vt = [&](int st) { return sm.base + (4 + st) * TILE; };
    const int col = h * HD;
    const int rowq = b * p.T + qb * BR;

    if (warp == 0 && lane == 0) {
        tc::mbar_expect_tx(qd_full, 2 * TILE);
        load_tile(Q, &mq, qd_full, col, rowq);
        load_tile(dO, &mdo, qd_full, col, rowq);
        for (int j = 0; j < nkb; ++j) {
            const int st = j & 1;
            const uint32_t ph = ((j >> 1) & 1) ^ 1;
            if (!tc::mbar_wait(&k_empty[st], ph, sm.abort)) break;
            tc::mbar_expect_tx(&k_full[st], TILE);
            load_tile(Kt(st), &mk, &k_full[st], col, b * p.T + j * BR);
            if (!tc::mbar_wait(&v_empty[st], ph, sm.abort)) break;
            tc::mbar_expect_tx(&v_full[st], TILE);
            load_tile(Vt(st), &mv, &v_full[st], col, b * p.T + j * BR);
        }
    } else if (warp == 1 && lane == 0) {
        const uint32_t q0 = tc::smem_u32(Q), do0 = tc::smem_u32(dO);
        // S and dP of block j (TMEM 0, 128) are read only by the softmax, so the next
        // block's S and dP go in as soon as the softmax is done with them (ds_full),
        // ahead of dQ_j: the softmax of block j+1 overlaps dQ_j
        auto issue_sdp = [&](int j) -> bool {
            const int st = j & 1;
            if (!tc::mbar_wait(&k_full[st], (j >> 1) & 1, sm.abort)) return false;
            tc::fence_after();
            const uint32_t k0 = tc::smem_u32(Kt(st)), v0 = tc::smem_u32(Vt(st));
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) tc::mma_bf16(tmem, dk_(q0, kk), dk_(k0, kk), IDESC_KK, kk > 0);
            if (!tc::mbar_wait(&v_full[st], (j >> 1) & 1, sm.abort)) return false;
            tc::fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) tc::mma_bf16(tmem + 128, dk_(do0, kk), dk_(v0, kk), IDESC_KK, kk > 0);
            tc::mma_commit(s_full);
            tc::mma_commit(&v_empty[st]);
            return true;
        };
        bool ok = tc::mbar_wait(qd_full, 0, sm.abort) && issue_sdp(0);
        for (int j = 0; ok && j < nkb; ++j) {
            const int st = j & 1;
            if (!(ok = tc::mbar_wait(ds_full, j & 1, sm.abort))) break;
            if (j + 1 < nkb && !(ok = issue_sdp(j + 1))) break;
            tc::fence_after();
            const uint32_t k0 = tc::smem_u32(Kt(st));
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                tc::mma_bf16_ts(tmem + 256, tmem + 384 + kk * 8, dm_(k0, kk), IDESC_KM, (j > 0 || kk > 0));
            tc::mma_commit(dq_done);
            tc::mma_commit(&k_empty[st]);
        }
    } else if (warp >= 2) {
        const int g = (warp - 2) >> 2, q = warp & 3, r = q * 32 + lane;
        const uint32_t lanes = (uint32_t)(q * 32) << 16;
        const float c2 = p.scale * LOG2E;
        const int t = qb * BR + r;
        const long st_i = ((long)b * p.H + h) * p.T + (t < p.T ? t : 0);
        const float lse2 = t < p.T ? p.lse[st_i] * LOG2E : INFINITY;
        const float Dt = t < p.T ? p.delta[st_i] : 0.f;
        float s[64];
        bool ok = true;
        for (int j = 0; j < nkb; ++j) {
            if (!(ok = tc::mbar_wait_warp(s_full, j & 1, sm.abort))) break;
            tc::fence_after();
            ld_half(tmem + lanes, g, s);
#pragma unroll
            for (int i = 0; i < 64; ++i) s[i] = exp2f(fmaf(s[i], c2, -lse2));
            if (j == qb) {
#pragma unroll
                for (int i = 0; i < 64; ++i)
                    if (col_of(g, i) > r) s[i] = 0.f;
            }
            uint32_t w[32];
            {
                float d[64];
                ld_half(tmem + lanes + 128, g, d);
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    w[i] = pack2(s[2 * i] * (d[2 * i] - Dt), s[2 * i + 1] * (d[2 * i + 1] - Dt));
            }
            // dS_{j-1} here was read by dQ_{j-1}; S_j was issued after ds_full_{j-1}
            // and dQ_{j-1} follows it, so wait for dQ_{j-1} before overwriting
            if (j > 0 && !(ok = tc::mbar_wait_warp(dq_done, (j - 1) & 1, sm.abort))) break;
            st_half_bf16(tmem + lanes + 384, g, w);
            tc::tmem_wait_st();
            tc::fence_before();
            tc::mbar_arrive(ds_full);
        }
        if (ok && tc::mbar_wait_warp(dq_done, (nkb - 1) & 1, sm.abort)) {
            tc::fence_after();
            ld_half(tmem + lanes + 256, g, s);
            if (t < p.T) {
                if (p.rope) unrope_half(s, p.rope, p.rope_ld, t, g);
                store_out_half(p.dq + (long)(b * p.T + t) * p.ldd + col, g, s, p.scale);
            }
        }
    }
    teardown(sm, tmem, p.flag);
}

// ===================================================================== dK, dV
// smem tiles: 0 K | 1 V | 2..4 Q stages | 5,6 dO stages
// barriers: 0 kv_full, 1-3 q_full, 4-6 q_empty, 7-8 do_full, 9-10 do_empty (one arrival
//           from each chain), 11 s_full, 12 dp_full, 14 p_full, 15 ds_full, 16 dv_done,
//           17 dk_done, 18-19 stat barriers
// TMEM: S^T at 0, dP^T at 128, dV at 256, dK at 384.  Each softmax group packs its bf16
// operands only into the columns it read itself (the two groups never wait for each
// other): P^T over S^T (group g at 32g .. 32g+31), dS^T over dP^T (at 192 + 32g ..); the
// products take each 16-query K slice from where its group left it (pk_col).  That gives
// two chains per query block, S^T -> P^T -> dV and dP^T -> dS^T -> dK, and each has an
// issuing thread of its own (warp 1 and the last warp).  A commit tracks only its own
// thread's products, and an issue that waits for a tensor-pipe slot holds back only its
// own chain, so P^T_i goes to dV_i as soon as it exists while dK_{i-1} or dP^T_i is still
// in the pipe.  Three Q stages let the loads run ahead.
constexpr int DKV_TILES = 7;
constexpr int DKV_QST = 3, DKV_DST = 2;
constexpr int DKV_NT = NT + 32;          // + the second issuing warp

// TMEM column (relative to the packed region) of K slice kk (queries 16kk .. 16kk+15)
// of a packed operand: queries [32g, 32g+32) and [64+32g, 64+32g+32) belong to group g,
// which stores them as 32 consecutive columns at 32g.
__host__ __device__ constexpr uint32_t pk_col(int kk) {
    return 32u * ((kk >> 1) & 1) + 16u * (kk >> 2) + 8u * (kk & 1);
}

__global__ void __launch_bounds__(DKV_NT, 1)
    attn_dkdv_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                     const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mdo,
                     const AttnParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    if (misaligned(smem_raw, p.flag)) return;
    Smem sm = carve(smem_raw, DKV_TILES);
    const int bh = blockIdx.y, kb = blockIdx.x, h = bh % p.H, b = bh / p.H;  // early keys (most work) first
    if (kb >= p.nblk) return;          // (a grid wider than the sequence: nothing to do)
    const int nq = p.nblk - kb;        // query blocks kb .. nblk-1
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    uint64_t* kv_full = &sm.bar[0];
    uint64_t* q_full = &sm.bar[1];
    uint64_t* q_empty = &sm.bar[4];
    uint64_t* do_full = &sm.bar[7];
    uint64_t* do_empty = &sm.bar[9];
    uint64_t* s_full = &sm.bar[11];
    uint64_t* dp_full = &sm.bar[12];
    uint64_t* p_full = &sm.bar[14];
    uint64_t* ds_full = &sm.bar[15];
    uint64_t* dv_done = &sm.bar[16];
    uint64_t* dk_done = &sm.bar[17];
    uint64_t* sbar = &sm.bar[18];
    const uint32_t counts[20] = {1, 1, 1, 1, 1, 1, 1, 1, 1, 2, 2, 1, 1, 1, NSM, NSM, 1, 1, NSM, NSM};
    setup(sm, 20, counts);
    const uint32_t tmem = *sm.tmem_slot;
    uint8_t* K = sm.base;
    uint8_t* V = sm.base + TILE;
    auto Qt = [&](int i) { return sm.base + (2 + i % DKV_QST) * TILE; };
    auto dOt = [&](int i) { return sm.base + (2 + DKV_QST + i % DKV_DST) * TILE; };
    const int col = h * HD;
    const int rowk = b * p.T + kb * BR;

    if (warp == 0 && lane == 0) {
        tc::mbar_expect_tx(kv_full, 2 * TILE);
        load_tile(K, &mk, kv_full, col, rowk);
        load_tile(V, &mv, kv_full, col, rowk);
        // Q runs up to three blocks ahead, dO two; interleave so neither starves the other
        int iq = 0, id = 0;
        bool ok = true;
        while (ok && (iq < nq || id < nq)) {
            if (iq < nq && iq <= id + 1) {
                const int st = iq % DKV_QST;
                if (!(ok = tc::mbar_wait(&q_empty[st], ((iq / DKV_QST) & 1) ^ 1, sm.abort))) break;
                tc::mbar_expect_tx(&q_full[st], TILE);
                load_tile(Qt(iq), &mq, &q_full[st], col, b * p.T + (kb + iq) * BR);
                ++iq;
            } else {
                const int st = id % DKV_DST;
                if (!(ok = tc::mbar_wait(&do_empty[st], ((id / DKV_DST) & 1) ^ 1, sm.abort))) break;
                tc::mbar_expect_tx(&do_full[st], TILE);
                load_tile(dOt(id), &mdo, &do_full[st], col, b * p.T + (kb + id) * BR);
                ++id;
            }
        }
    } else if (warp == 1 && lane == 0) {
        // chain one: S^T_i = K Q_i^T, then dV += P^T_i dO_i (P^T_i packed over S^T_i)
        const uint32_t k0 = tc::smem_u32(K);
        bool ok = tc::mbar_wait(kv_full, 0, sm.abort);
        for (int i = 0; ok && i < nq; ++i) {
            const uint32_t qn = tc::smem_u32(Qt(i)), do0 = tc::smem_u32(dOt(i));
            // S^T_i overwrites P^T_{i-1}, which dV_{i-1} reads: that product has completed
            if (i > 0 && !(ok = tc::mbar_wait(dv_done, (i - 1) & 1, sm.abort))) break;
            if (!(ok = tc::mbar_wait(&q_full[i % DKV_QST], (i / DKV_QST) & 1, sm.abort))) break;
            tc::fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) tc::mma_bf16(tmem, dk_(k0, kk), dk_(qn, kk), IDESC_KK, kk > 0);
            tc::mma_commit(s_full);
            if (!(ok = tc::mbar_wait(p_full, i & 1, sm.abort))) break;
            tc::fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                tc::mma_bf16_ts(tmem + 256, tmem + pk_col(kk), dm_(do0, kk), IDESC_KM, (i > 0 || kk > 0));
            tc::mma_commit(dv_done);
            tc::mma_commit(&do_empty[i % DKV_DST]);
        }
    } else if (warp == DKV_NT / 32 - 1 && lane == 0) {
        // chain two: dP^T_i = V dO_i^T, then dK += dS^T_i Q_i (dS^T_i packed over dP^T_i)
        const uint32_t v0 = tc::smem_u32(V);
        bool ok = tc::mbar_wait(kv_full, 0, sm.abort);
        for (int i = 0; ok && i < nq; ++i) {
            const uint32_t q0 = tc::smem_u32(Qt(i)), don = tc::smem_u32(dOt(i));
            // dP^T_i overwrites dS^T_{i-1}, which dK_{i-1} reads: that product has completed
            if (i > 0 && !(ok = tc::mbar_wait(dk_done, (i - 1) & 1, sm.abort))) break;
            if (!(ok = tc::mbar_wait(&do_full[i % DKV_DST], (i / DKV_DST) & 1, sm.abort))) break;
            tc::fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) tc::mma_bf16(tmem + 128, dk_(v0, kk), dk_(don, kk), IDESC_KK, kk > 0);
            tc::mma_commit(dp_full);
            tc::mma_commit(&do_empty[i % DKV_DST]);
            // Q_i: S^T_i has completed (the softmax read it before dS^T_i exists)
            if (!(ok = tc::mbar_wait(ds_full, i & 1, sm.abort))) break;
            tc::fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                tc::mma_bf16_ts(tmem + 384, tmem + 192 + pk_col(kk), dm_(q0, kk), IDESC_KM, (i > 0 || kk > 0));
            tc::mma_commit(dk_done);
            tc::mma_commit(&q_empty[i % DKV_QST]);
        }
    } else if (warp >= 2 && warp < 10) {
        const int g = (warp - 2) >> 2, q = warp & 3, r = q * 32 + lane;   // r = key row of the block
        const uint32_t lanes = (uint32_t)(q * 32) << 16;
        const float c2 = p.scale * LOG2E;
        const long srow = ((long)b * p.H + h) * p.T;
        // this thread's statistic of query row kb*BR + 128 i + r (group 0: lse, 1: D),
        // loaded one block ahead so its latency hides under the previous block
        const float* src = (g == 0 ? p.lse : p.delta) + srow;
        auto fetch = [&](int jb) { const int t = jb * BR + r; return t < p.T ? src[t] : NAN; };
        float nxt = fetch(kb);
        // publish query block i's statistics: [-lse2 | -D] in exchange buffer i % 2
        auto put_stat = [&](int i) {
            const int j = kb + i;
            float* stat = sm.xch + (i & 1) * 256;
            const float cur = nxt;
            if (i + 1 < nq) nxt = fetch(j + 1);
            const bool valid = j * BR + r < p.T;
            if (g == 0) stat[r] = valid ? -cur * LOG2E : -INFINITY;
            else stat[128 + r] = valid ? -cur : 0.f;
            tc::mbar_arrive(&sbar[i & 1]);
        };
        put_stat(0);
        float s[64];
        bool ok = true;
        for (int i = 0; i < nq; ++i) {
            const int j = kb + i;
            const float* stat = sm.xch + (i & 1) * 256;
            if (!(ok = tc::mbar_wait_warp(&sbar[i & 1], (i >> 1) & 1, sm.abort))) break;
            if (!(ok = tc::mbar_wait_warp(s_full, i & 1, sm.abort))) break;
            tc::fence_after();
            ld_half(tmem + lanes, g, s);
            // P^T[r][c] = exp2(S^T*c2 - lse2[c]), zero where key r > query c; this
            // thread's columns are two contiguous runs of 32 (statistics as pairs), the
            // scale and shift two lanes at a time
            const uint64_t c22 = tc::f2pk(c2, c2);
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                // (16-byte broadcast loads: shared memory is the tensor core's operand path)
                const float4* l4 = reinterpret_cast<const float4*>(stat + 64 * h2 + 32 * g);
#pragma unroll
                for (int k4 = 0; k4 < 8; ++k4) {
                    const float4 l = l4[k4];
                    float* x = s + 32 * h2 + 4 * k4;
                    float a, bb;
                    tc::f2upk(tc::ffma2(tc::f2pk(x[0], x[1]), c22, tc::f2pk(l.x, l.y)), a, bb);
                    x[0] = tc::ex2a(a);
                    x[1] = tc::ex2a(bb);
                    tc::f2upk(tc::ffma2(tc::f2pk(x[2], x[3]), c22, tc::f2pk(l.z, l.w)), a, bb);
                    x[2] = tc::ex2a(a);
                    x[3] = tc::ex2a(bb);
                }
            }
            if (i == 0) {
#pragma unroll
                for (int e = 0; e < 64; ++e)
                    if (r > col_of(g, e)) s[e] = 0.f;
            }
            {   // P^T into this group's S^T columns (already read): dV_i can start now
                uint32_t wp[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) wp[e] = pack2(s[2 * e], s[2 * e + 1]);
                tc::tmem_st32(tmem + lanes + 32 * g, wp);
                tc::tmem_wait_st();
                tc::fence_before();
                tc::mbar_arrive(p_full);
            }
            uint32_t wd[32];
            {
                uint32_t d[32];   // this thread's dP^T, one 32-query chunk at a time
                if (!(ok = tc::mbar_wait_warp(dp_full, i & 1, sm.abort))) break;
                tc::fence_after();
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {   // dS^T = P^T (dP^T - D[c])
                    tc::tmem_ld32(tmem + lanes + 128 + 64 * h2 + 32 * g, d);
                    tc::tmem_wait_ld();
                    const float4* nd4 = reinterpret_cast<const float4*>(stat + 128 + 64 * h2 + 32 * g);
#pragma unroll
                    for (int k4 = 0; k4 < 8; ++k4) {   // (dP^T - D) * P^T, two lanes at a time
                        const float4 nd = nd4[k4];
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            const int k2 = 2 * k4 + u;
                            const float* x = s + 32 * h2 + 2 * k2;
                            const uint32_t* y = d + 2 * k2;
                            float a, bb;
                            tc::f2upk(tc::fmul2(tc::f2pk(x[0], x[1]),
                                        tc::fadd2(tc::f2pk(__uint_as_float(y[0]), __uint_as_float(y[1])),
                                                  u ? tc::f2pk(nd.z, nd.w) : tc::f2pk(nd.x, nd.y))),
                                  a, bb);
                            wd[16 * h2 + k2] = pack2(a, bb);
                        }
                    }
                }
            }
            tc::tmem_st32(tmem + lanes + 192 + 32 * g, wd);
            tc::tmem_wait_st();
            tc::fence_before();
            tc::mbar_arrive(ds_full);
            // the next block's statistics go out before this block's dS store, so that no
            // thread waits on another's stores (every thread has read buffer (i+1) % 2,
            // block i-1's, since the barrier of block i)
            if (i + 1 < nq) put_stat(i + 1);
            if (p.ds) {   // keep key r's dS for the dQ product: query chunks 4g+k and 8+4g+k
                uint8_t* base = ds_tile(p, bh, j, kb) + (r >> 6) * DS_HALF + (r & 63) * 16;
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint32_t* x = wd + 16 * h2 + 4 * k;
                        *reinterpret_cast<uint4*>(base + (8 * h2 + 4 * g + k) * 1024) =
                            make_uint4(x[0], x[1], x[2], x[3]);
                    }
            }
        }
        if (ok && tc::mbar_wait_warp(dk_done, (nq - 1) & 1, sm.abort) &&
            tc::mbar_wait_warp(dv_done, (nq - 1) & 1, sm.abort)) {
            tc::fence_after();
            const int key = kb * BR + r;
            ld_half(tmem + lanes + 256, g, s);
            if (key < p.T) store_out_half(p.dv + (long)(b * p.T + key) * p.ldd + col, g, s, 1.f);
            ld_half(tmem + lanes + 384, g, s);
            if (key < p.T) {
                if (p.rope) unrope_half(s, p.rope, p.rope_ld, key, g);
                store_out_half(p.dk + (long)(b * p.T + key) * p.ldd + col, g, s, p.scale);
            }
        }
    }
    teardown(sm, tmem, p.flag);
}

// ===================================================================== dQ from the dS^T store
// dQ_i = scale * sum_{j<=i} dS_ij K_j as a streamed block-causal product: the dK/dV
// kernel has already formed every dS_ij, so nothing is recomputed here.  Stages hold
// 64 keys: the stored dS half (64 keys x 128 queries, the interleaved MN-major A
// operand, one plain bulk copy) and the K half-tile (64 keys x 128 dims, the
// 128-byte-swizzled MN-major B operand, by TMA).  Four warps read dQ out of
// TMEM; two CTAs share an SM so one's epilogue overlaps the other's stream.
// barriers: 0..2 full, 3..5 empty, 6 done, 7 drain
constexpr int DQS_NT = 192;              // producer warp, MMA warp, 4 epilogue warps
constexpr int HATOM = 64 * 128;          // 8 KB: 64 rows x 64 bf16, 128-byte swizzle
constexpr int DQS_ST = 3;                // stages of 4 atoms (one TILE) each
constexpr uint32_t IDESC_MM = tc::idesc_bf16(128, 128, true, true);

// MN-major view of a 64-row half tile (MN = its 128 columns, two atoms), k-th 16-row slice
__device__ __forceinline__ uint64_t dh_(uint32_t half, int kk) { return tc::sdesc(half + kk * 2048, HATOM, 1024); }
// the stored dS half (interleaved MN-major: 8-key groups 128 B apart, 8-query chunks 1 KB apart)
__device__ __forceinline__ uint64_t dsa_(uint32_t half, int kk) { return tc::sdesc_none(half + kk * 256, 128, 1024); }

__global__ void __launch_bounds__(DQS_NT, 2)
    attn_dq_ds_kernel(const __grid_constant__ CUtensorMap mk, const AttnParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    if (misaligned(smem_raw, p.flag)) return;
    Smem sm = carve(smem_raw, DQS_ST);
    const int bh = blockIdx.y, qb = p.nblk - 1 - (int)blockIdx.x, h = bh % p.H, b = bh / p.H;
    if (qb < 0) return;                // (a grid wider than the sequence: nothing to do)
    const int nu = 2 * (qb + 1);           // 64-key units up to the diagonal
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    uint64_t* full = &sm.bar[0];
    uint64_t* empty = &sm.bar[3];
    uint64_t* done = &sm.bar[6];
    uint64_t* drain = &sm.bar[7];
    const uint32_t counts[8] = {1, 1, 1, 1, 1, 1, 1, 1};
    setup(sm, 8, counts, 128);
    const uint32_t tmem = *sm.tmem_slot;
    const int col = h * HD;

    if (warp == 0 && lane == 0) {
        const uint8_t* ds0 = ds_tile(p, bh, qb, 0);
        int u = 0;
        for (; u < nu; ++u) {
            const int st = u % DQS_ST;
            if (!tc::mbar_wait(&empty[st], ((u / DQS_ST) & 1) ^ 1, sm.abort)) break;
            uint8_t* dst = sm.base + st * TILE;
            tc::mbar_expect_tx(&full[st], TILE);
            const int kr = b * p.T + 64 * u;
            tc::bulk_load(dst, ds0 + (long)u * DS_HALF, DS_HALF, &full[st]);
            tc::tma_load_3d(dst + 2 * HATOM, &mk, &full[st], col, kr, 0);
            tc::tma_load_3d(dst + 3 * HATOM, &mk, &full[st], col + 64, kr, 0);
        }
        if (*sm.abort)   // let the copies still in flight land before the CTA exits
            for (int w = u - 1; w >= 0 && w >= u - DQS_ST; --w)
                tc::mbar_wait_drain(&full[w % DQS_ST], (w / DQS_ST) & 1);
    } else if (warp == 1 && lane == 0) {
        bool ok = true;
        for (int u = 0; u < nu; ++u) {
            const int st = u % DQS_ST;
            if (!(ok = tc::mbar_wait(&full[st], (u / DQS_ST) & 1, sm.abort))) break;
            tc::fence_after();
            const uint32_t a0 = tc::smem_u32(sm.base + st * TILE), b0 = a0 + 2 * HATOM;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) tc::mma_bf16(tmem, dsa_(a0, kk), dh_(b0, kk), IDESC_MM, (u > 0 || kk > 0));
            tc::mma_commit(&empty[st]);
        }
        if (ok) tc::mma_commit(done);
        if (*sm.abort) {
            tc::mma_commit(drain);
            tc::mbar_wait_drain(drain, 0);
        }
    } else if (warp >= 2) {
        const int q = warp & 3, r = q * 32 + lane;
        const uint32_t lanes = (uint32_t)(q * 32) << 16;
        const int t = qb * BR + r;
        if (tc::mbar_wait_warp(done, 0, sm.abort)) {
            tc::fence_after();
            float v[64];
#pragma unroll 1
            for (int g = 0; g < 2; ++g) {
                ld_half(tmem + lanes, g, v);
                if (t < p.T) {
                    if (p.rope) unrope_half(v, p.rope, p.rope_ld, t, g);
                    store_out_half(p.dq + (long)(b * p.T + t) * p.ldd + col, g, v, p.scale);
                }
            }
        }
    }
    teardown(sm, tmem, p.flag, 128);
}

int smem_bytes(int tiles) { return tiles * TILE + 256 + XCH_BYTES; }

template <typename K>
int set_smem(K kern, int bytes) {
    return cuda_check(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes),
                      "attention smem attribute");
}

int maps(CUtensorMap* m, const void* ptr, long rows, long ld, int H) {
    return make_map(m, ptr, (long)H * HD, rows, 1, ld, 0, 64, BR);
}

}  // namespace

// Grids are (blocks of a sequence, batch x heads): the x index runs fastest, so the
// CTAs of one batch-head are resident together and share its K/V (forward, dQ) or
// Q/dO (dK/dV) tiles through L2 instead of re-reading them from HBM.
constexpr long MAX_GRID_Y = 65535;

bool attention_tc_supported(long ld, long ldo, long ldd, const void* q, const void* k, const void* v,
                            int D) {
    if (D != HD) return false;
    if (ld % 8 || ldo % 8 || ldd % 8) return false;
    if ((uintptr_t)q % 16 || (uintptr_t)k % 16 || (uintptr_t)v % 16) return false;
    return true;
}

int attention_forward_tc(const bf16* q, const bf16* k, const bf16* v, long ld, bf16* o, long ldo,
                         float* lse, int B, int T, int H, cudaStream_t s, uint32_t* flag) {
    if ((long)B * H > MAX_GRID_Y) return set_error(NC_ERR_UNSUPPORTED, "attention: B*H = %ld > %ld", (long)B * H, MAX_GRID_Y);
    static DeviceOnce init;
    NC_TRY(init.run([] { return set_smem(attn_fwd_kernel, smem_bytes(FWD_TILES)); }));
    CUtensorMap mq, mk, mv;
    const long rows = (long)B * T;
    NC_TRY(maps(&mq, q, rows, ld, H));
    NC_TRY(maps(&mk, k, rows, ld, H));
    NC_TRY(maps(&mv, v, rows, ld, H));
    AttnParams p{};
    p.T = T; p.H = H; p.nblk = ceil_div(T, BR); p.ldo = ldo; p.o = o; p.lse = lse;
    p.scale = 1.0f / sqrtf((float)HD); p.flag = flag;
    attn_fwd_kernel<<<dim3((p.nblk + 1) / 2, H * B), NT, smem_bytes(FWD_TILES), s>>>(mq, mk, mv, p);
    note_launch();
    NC_LAUNCH_CHECK("attn_fwd_kernel");
    return NC_OK;
}

// dS store: B*H*nblk(nblk+1)/2 tiles of 128 x 128 bf16
size_t attention_tc_ds_bytes(int B, int T, int H) {
    const long nblk = ceil_div(T, BR);
    return (size_t)B * H * (nblk * (nblk + 1) / 2) * DS_TILE;
}

int attention_backward_tc(const bf16* q, const bf16* k, const bf16* v, long ld, const bf16* dout,
                          long ldo, const float* lse, const float* delta, bf16* dq, bf16* dk, bf16* dv,
                          long ldd, int B, int T, int H, const float2* rope, int rope_ld, bf16* ds,
                          cudaStream_t s, uint32_t* flag) {
    if ((long)B * H > MAX_GRID_Y) return set_error(NC_ERR_UNSUPPORTED, "attention: B*H = %ld > %ld", (long)B * H, MAX_GRID_Y);
    static DeviceOnce init;
    NC_TRY(init.run([] {
        NC_TRY(set_smem(attn_dq_kernel, smem_bytes(DQ_TILES)));
        NC_TRY(set_smem(attn_dkdv_kernel, smem_bytes(DKV_TILES)));
        return set_smem(attn_dq_ds_kernel, smem_bytes(DQS_ST));
    }));
    if ((uintptr_t)ds % 16) ds = nullptr;
    CUtensorMap mq, mk, mv, mdo;
    const long rows = (long)B * T;
    NC_TRY(maps(&mq, q, rows, ld, H));
    NC_TRY(maps(&mk, k, rows, ld, H));
    NC_TRY(maps(&mv, v, rows, ld, H));
    NC_TRY(maps(&mdo, dout, rows, ldo, H));
    AttnParams p{};
    p.T = T; p.H = H; p.nblk = ceil_div(T, BR); p.ldo = ldo; p.ldd = ldd;
    p.lse = const_cast<float*>(lse); p.delta = delta; p.dq = dq; p.dk = dk; p.dv = dv; p.rope = rope;
    p.rope_ld = rope_ld;
    p.scale = 1.0f / sqrtf((float)HD); p.flag = flag;
    p.ds = ds; p.ds_bh = (long)p.nblk * (p.nblk + 1) / 2;
    attn_dkdv_kernel<<<dim3(p.nblk, H * B), DKV_NT, smem_bytes(DKV_TILES), s>>>(mq, mk, mv, mdo, p);
    if (ds) {
        CUtensorMap mk64;
        NC_TRY(make_map(&mk64, k, (long)H * HD, rows, 1, ld, 0, 64, 64));
        attn_dq_ds_kernel<<<dim3(p.nblk, H * B), DQS_NT, smem_bytes(DQS_ST), s>>>(mk64, p);
    } else {
        attn_dq_kernel<<<dim3(p.nblk, H * B), NT, smem_bytes(DQ_TILES), s>>>(mq, mk, mv, mdo, p);
    }
    note_launch(2);
    NC_LAUNCH_CHECK("attn backward kernels");
    return NC_OK;
}

}  // namespace nc
