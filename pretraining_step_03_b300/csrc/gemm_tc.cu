// bf16 GEMM on the 5th-generation tensor cores (tcgen05 + TMEM, TMA-fed).
//
// C = alpha * op(A) op(B)^T with the step's fused epilogues (residual add,
// ReLU^2 forward/backward, axpby, fp32/bf16 stores).  It serves every dense
// contraction of the step: the q|k|v, attention-output, MLP and LM-head
// projections (nanochat speedrun walkthrough, lyylswood.com, section 预搜检:
// 1280 channels, 4x MLP at d20), their two backward products, and the
// batched Newton-Schulz matmuls of Muon.
//
// Design (one CTA per SM, persistent over output tiles):
//   warp 0      TMA producer: A and B k-slices (64 wide, 128-byte swizzle)
//               into a ring of shared-memory stages;
//   warp 1      allocates TMEM and issues tcgen05.mma (M=128, N=BN, K=16)
//               from one thread; commits free smem stages and finished
//               accumulators;
//   warps 2-5   epilogue: tcgen05.ld of the fp32 accumulator (one row per
//               thread), fused elementwise work, vector stores.
// The accumulator is double-buffered in TMEM (2 x BN columns) so the
// epilogue of one tile overlaps the MMAs of the next.  Operands can be
// K-major or MN-major, so backward products read activations and weights
// in place (no transposes).  Small-output GEMMs (weight gradients) split K
// over CTAs into an fp32 scratch and reduce in a fixed order.
#include <cudaTypedefs.h>

#include <mutex>

#include "kernels.cuh"
#include "tc_ptx.cuh"

namespace nc {
namespace {

constexpr int BM = 128, BK = 64, NTHREADS = 320, GROUP_M = 8;
constexpr int EPI_WARPS = 8;   // two groups of four, each owns half the tile columns
// Per epilogue warp: 8 KB holding a ring of 32 x 32 blocks laid out with the 128-byte
// (fp32, 4 KB) / 64-byte (bf16, 2 KB) TMA swizzle: two fp32 or four bf16 slots.  They
// receive the auxiliary matrix by TMA, a whole tile's chunks ahead where they fit, and
// then serve as the staging of the coalesced store.
constexpr int EPI_BUF = 4096;
constexpr int EPI_STG = 2 * EPI_BUF;
constexpr int XSLOTS_MAX = 4;
constexpr int EPI_STG_BYTES = EPI_WARPS * EPI_STG;
constexpr int BAR_BYTES = 512;   // mbarriers, TMEM slot, abort flag (after the staging)

struct TcParams {
    int M, N, K, batch;
    int tiles_m, tiles_n, splits, num_kb;
    long units;
    void* C; long ldc, sC; int c_dtype;
    const void* aux; long ldaux, sAux; int aux_dtype;
    float alpha, beta;
    int epi;
    float* ws;        // split-K partials [splits][batch][M][N], or null
    uint32_t* flag;   // device flag word for timeouts (may be null)
    const float2* rope;   // (cos, sin) of pair j at position t: rope[j * rope_ld + t]
    int rope_T, rope_cols, rope_ld;
    float* delta;
    int aux_tma;      // the auxiliary matrix comes through the per-warp TMA buffers
    int sym;          // symmetric C: upper-triangle tiles only, mirrored (tiles_m == tiles_n)
    float2* lse_part; // EPI_LSE: [M][N/128] (max, sum exp) partials
    float* dot_out;       // EPI_RELU2_BWD: [M][N/128] <dh, relu(h)> partials (may be null)
    const float* nb_r;    // EPI_NORMB: rstd [M], row-dot partials [M][nb_nparts], 1/d,
    const float* nb_part; //   residual gradient in (fp32, C's layout; may alias C), bf16 copy out
    int nb_nparts;
    float nb_inv_d;
    const float* nb_gin;
    bf16* nb_gt;
};

template <int BN> struct Cfg {
    static constexpr int A_BYTES = BM * BK * 2;
    static constexpr int B_BYTES = BN * BK * 2;
    static constexpr int STAGE = A_BYTES + B_BYTES;
    static constexpr int STAGES = BN == 256 ? 3 : 4;
    static constexpr uint32_t TMEM_COLS = 2 * BN;
    static constexpr int SMEM = STAGES * STAGE + 1024 + BAR_BYTES + EPI_STG_BYTES;
};

__device__ __forceinline__ void decode(const TcParams& p, long u, int& b, int& split, int& tm,
                                       int& tn) {
    if (p.sym) {   // tiles (tm, tn), tn >= tm, row by row
        const long tiles = (long)p.tiles_m * (p.tiles_m + 1) / 2;
        long t = u % tiles;
        b = (int)(u / tiles);
        split = 0;
        int i = 0;
        while (t >= p.tiles_m - i) { t -= p.tiles_m - i; ++i; }
        tm = i;
        tn = i + (int)t;
        return;
    }
    const long tiles = (long)p.tiles_m * p.tiles_n;
    const long t = u % tiles, bs = u / tiles;
    split = (int)(bs % p.splits);
    b = (int)(bs / p.splits);
    const long per_group = (long)GROUP_M * p.tiles_n;
    const int g = (int)(t / per_group);
    const int first_m = g * GROUP_M;
    const int gsize = min(p.tiles_m - first_m, GROUP_M);
    const int r = (int)(t % per_group);
    tm = first_m + r % gsize;
    tn = r / gsize;
}

__device__ __forceinline__ void kb_range(const TcParams& p, int split, int& kb0, int& kb1) {
    kb0 = (int)((long)split * p.num_kb / p.splits);
    kb1 = (int)((long)(split + 1) * p.num_kb / p.splits);
}

__device__ __forceinline__ float ld_elem(const void* base, long i, int dt) {
    return dt == NC_FP32 ? reinterpret_cast<const float*>(base)[i]
                         : __bfloat162float(reinterpret_cast<const bf16*>(base)[i]);
}

// load 32 consecutive elements (16-byte aligned) as fp32
__device__ __forceinline__ void ld32(const void* base, long i, int dt, float* v) {
    if (dt == NC_FP32) {
        const float4* s = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(base) + i);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            float4 f = s[j];
            v[4 * j] = f.x; v[4 * j + 1] = f.y; v[4 * j + 2] = f.z; v[4 * j + 3] = f.w;
        }
    } else {
        const uint4* s = reinterpret_cast<const uint4*>(reinterpret_cast<const bf16*>(base) + i);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint4 u = s[j];
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162*>(&w[e]);
                float2 f = __bfloat1622float2(h);
                v[8 * j + 2 * e] = f.x;
                v[8 * j + 2 * e + 1] = f.y;
            }
        }
    }
}

__device__ __forceinline__ void st32(void* base, long i, int dt, const float* v) {
    if (dt == NC_FP32) {
        float4* d = reinterpret_cast<float4*>(reinterpret_cast<float*>(base) + i);
#pragma unroll
        for (int j = 0; j < 8; ++j) d[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    } else {
        uint4* d = reinterpret_cast<uint4*>(reinterpret_cast<bf16*>(base) + i);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                __nv_bfloat162 h = __floats2bfloat162_rn(v[8 * j + 2 * e], v[8 * j + 2 * e + 1]);
                w[e] = *reinterpret_cast<uint32_t*>(&h);
            }
            d[j] = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
}

__device__ __forceinline__ void st_elem(void* base, long i, int dt, float v) {
    if (dt == NC_FP32) reinterpret_cast<float*>(base)[i] = v;
    else reinterpret_cast<bf16*>(base)[i] = __float2bfloat16_rn(v);
}

// bf16 rows already rounded and packed (word k = columns 2k, 2k+1): the store side of
// wst32's bf16 path, and the per-lane form.
__device__ __forceinline__ void wst32_bf16w(uint8_t* stg, void* base, long off0, long ld, const uint32_t* w) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int c = 0; c < 4; ++c)
        *reinterpret_cast<uint4*>(stg + lane * 64 + ((c ^ ((lane >> 1) & 3)) << 4)) =
            make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
    __syncwarp();
    bf16* out = reinterpret_cast<bf16*>(base) + off0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = 8 * i + (lane >> 2), c = lane & 3;
        *reinterpret_cast<uint4*>(out + (long)r * ld + 8 * c) =
            *reinterpret_cast<const uint4*>(stg + r * 64 + ((c ^ ((r >> 1) & 3)) << 4));
    }
    __syncwarp();
}
__device__ __forceinline__ void st32_bf16w(void* base, long i, const uint32_t* w) {
    uint4* d = reinterpret_cast<uint4*>(reinterpret_cast<bf16*>(base) + i);
#pragma unroll
    for (int c = 0; c < 4; ++c) d[c] = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
}
// Rounds x, y to bf16, packs them (x in the low half) and returns the rounded values.
__device__ __forceinline__ uint32_t round_pack2(float& x, float& y) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
    const float2 f = __bfloat1622float2(h);
    x = f.x;
    y = f.y;
    return *reinterpret_cast<const uint32_t*>(&h);
}

// Warp-cooperative row I/O.  Lane i holds 32 consecutive columns of row r0 + i
// (rows ld elements apart, lane 0's first element at off0).  Going through the
// warp's staging buffer (swizzled by 16-byte chunk, conflict-free), every global
// access instruction covers whole 128-byte (fp32) or 64-byte (bf16) row segments,
// instead of 32 separate 16-byte pieces of 32 rows.
__device__ __forceinline__ void wst32(uint8_t* stg, void* base, long off0, long ld, int dt, const float* v) {
    const int lane = threadIdx.x & 31;
    if (dt == NC_FP32) {
#pragma unroll
        for (int c = 0; c < 8; ++c)
            *reinterpret_cast<float4*>(stg + lane * 128 + ((c ^ (lane & 7)) << 4)) =
                make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
        __syncwarp();
        float* out = reinterpret_cast<float*>(base) + off0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int r = 4 * i + (lane >> 3), c = lane & 7;
            *reinterpret_cast<float4*>(out + (long)r * ld + 4 * c) =
                *reinterpret_cast<const float4*>(stg + r * 128 + ((c ^ (r & 7)) << 4));
        }
        __syncwarp();
    } else {
        uint32_t w[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * k], v[2 * k + 1]);
            w[k] = *reinterpret_cast<uint32_t*>(&h);
        }
        wst32_bf16w(stg, base, off0, ld, w);
    }
}

// Pieces of wst32's bf16 path: stage_bf16x16 puts 16 values (columns 16h..16h+15)
// of this lane's row into a 32 x 32 bf16 staging block; flush_bf16 writes the
// block out (rows ld elements apart, lane 0's row at off0).
__device__ __forceinline__ void stage_bf16x16(uint8_t* stg, int h, const float* v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int c2 = 0; c2 < 2; ++c2) {
        const int c = 2 * h + c2;
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            __nv_bfloat162 x = __floats2bfloat162_rn(v[8 * c2 + 2 * e], v[8 * c2 + 2 * e + 1]);
            w[e] = *reinterpret_cast<uint32_t*>(&x);
        }
        *reinterpret_cast<uint4*>(stg + lane * 64 + ((c ^ ((lane >> 1) & 3)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}
__device__ __forceinline__ void flush_bf16(const uint8_t* stg, void* base, long off0, long ld) {
    const int lane = threadIdx.x & 31;
    __syncwarp();
    bf16* out = reinterpret_cast<bf16*>(base) + off0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = 8 * i + (lane >> 2), c = lane & 3;
        *reinterpret_cast<uint4*>(out + (long)r * ld + 8 * c) =
            *reinterpret_cast<const uint4*>(stg + r * 64 + ((c ^ ((r >> 1) & 3)) << 4));
    }
    __syncwarp();
}
__device__ __forceinline__ void st16_bf16(bf16* dst, const float* v) {
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            __nv_bfloat162 x = __floats2bfloat162_rn(v[8 * c + 2 * e], v[8 * c + 2 * e + 1]);
            w[e] = *reinterpret_cast<uint32_t*>(&x);
        }
        reinterpret_cast<uint4*>(dst)[c] = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// fp32 rows out through a 2 KB staging block, 16 columns at a time (64-byte rows laid
// out as the bf16 blocks above): lane i's 16 values of row r0 + i, rows ld elements
// apart, lane 0's first element at off0.
__device__ __forceinline__ void wst16_f32(uint8_t* stg, float* base, long off0, long ld, const float* v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int c = 0; c < 4; ++c)
        *reinterpret_cast<float4*>(stg + lane * 64 + ((c ^ ((lane >> 1) & 3)) << 4)) =
            make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
    __syncwarp();
    float* out = base + off0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = 8 * i + (lane >> 2), c = lane & 3;
        *reinterpret_cast<float4*>(out + (long)r * ld + 4 * c) =
            *reinterpret_cast<const float4*>(stg + r * 64 + ((c ^ ((r >> 1) & 3)) << 4));
    }
    __syncwarp();
}

// The auxiliary-matrix pipeline of one epilogue warp: 32 x 32 blocks come in by TMA
// into a ring of slots (two of 4 KB for fp32, four of 2 KB for bf16), consumed in
// issue order.  Kept in three registers: the buffer's and the barriers' shared
// addresses and a packed state word.
struct XPipe {
    uint32_t buf;       // shared address of the 8 KB ring
    uint32_t bar;       // shared address of XSLOTS_MAX mbarriers (arrival count 1)
    uint32_t st;        // bits 0-1 issue slot, 2-3 head slot, 4-7 phases, 8-11 pending, 12 fp32
    __device__ __forceinline__ int slots() const { return (st >> 12) & 1 ? 2 : 4; }
    __device__ __forceinline__ uint32_t bytes() const { return (st >> 12) & 1 ? 4096u : 2048u; }
    __device__ __forceinline__ uint64_t* barp(int k) const {
        return reinterpret_cast<uint64_t*>(__cvta_shared_to_generic(bar + 8 * k));
    }
    __device__ __forceinline__ uint8_t* bufp(int k) const {
        return reinterpret_cast<uint8_t*>(__cvta_shared_to_generic(buf + k * bytes()));
    }
};

__device__ __forceinline__ XPipe x_make(uint8_t* buf, uint64_t* bar, bool f32) {
    return XPipe{tc::smem_u32(buf), tc::smem_u32(bar), f32 ? 1u << 12 : 0u};
}

__device__ __forceinline__ void x_issue(XPipe& x, const CUtensorMap* m, int n0, int row0, int b) {
    const int k = x.st & 3;
    const int nk = k + 1 == x.slots() ? 0 : k + 1;
    x.st = (x.st & ~3u) | nk | (1u << (8 + k));
    __syncwarp();   // every lane is done with slot k (aux read or store staging)
    if ((threadIdx.x & 31) == 0) {
        tc::fence_async_smem();   // those generic-proxy accesses before the TMA write
        tc::mbar_expect_tx(x.barp(k), x.bytes());
        tc::tma_load_3d(x.bufp(k), m, x.barp(k), n0, row0, b);
    }
}

// The tile this epilogue warp handles next.  A warp's aux blocks are fetched in one
// sequence, this tile's chunks and then the next tile's, keeping the ring full: so the
// next tile's first blocks come in while this tile's last chunks are processed, instead
// of being waited for at the start of the next epilogue.
struct NextTile {
    bool on;       // there is a next tile and the aux matrix comes by TMA
    int tn, row, b;
    int next;      // index in that sequence of the next block to fetch (this tile: 0 .. n-1)
};

// A ring slot has just been freed: fetch the next block of the sequence, if any.
__device__ __forceinline__ void x_ahead(XPipe& x, const CUtensorMap* m, int cstart, int cend, int BN, int tn,
                                        int row, int b, NextTile& nt) {
    const int lane = threadIdx.x & 31, n = cend - cstart, j = nt.next;
    if (j < n) x_issue(x, m, tn * BN + (cstart + j) * 32, row - lane, b);
    else if (nt.on && j - n < n) x_issue(x, m, nt.tn * BN + (cstart + j - n) * 32, nt.row - lane, nt.b);
    else return;
    nt.next = j + 1;
}

// The oldest outstanding block, once it has landed (null if the CTA aborted).
__device__ __forceinline__ uint8_t* x_wait(XPipe& x, volatile int* abort) {
    const int k = (x.st >> 2) & 3;
    if (!tc::mbar_wait_warp(x.barp(k), (x.st >> (4 + k)) & 1, abort)) return nullptr;
    const int nk = k + 1 == x.slots() ? 0 : k + 1;
    x.st = ((x.st & ~(3u << 2)) | (nk << 2)) ^ (1u << (4 + k));
    x.st &= ~(1u << (8 + k));
    return x.bufp(k);
}

// After an abort: let issued copies land before the CTA exits.
__device__ __forceinline__ void x_drain(XPipe& x) {
    if ((threadIdx.x & 31) != 0) return;
    for (int k = 0; k < x.slots(); ++k)
        if ((x.st >> (8 + k)) & 1) tc::mbar_wait_drain(x.barp(k), (x.st >> (4 + k)) & 1);
}

// This lane's 32 values of a TMA-loaded block (the layout of wst32's staging).
__device__ __forceinline__ void x_row(const uint8_t* xb, int dt, float* a) {
    const int lane = threadIdx.x & 31;
    if (dt == NC_FP32) {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const float4 f = *reinterpret_cast<const float4*>(xb + lane * 128 + ((c ^ (lane & 7)) << 4));
            a[4 * c] = f.x; a[4 * c + 1] = f.y; a[4 * c + 2] = f.z; a[4 * c + 3] = f.w;
        }
    } else {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint4 u = *reinterpret_cast<const uint4*>(xb + lane * 64 + ((c ^ ((lane >> 1) & 3)) << 4));
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[e]));
                a[8 * c + 2 * e] = f.x;
                a[8 * c + 2 * e + 1] = f.y;
            }
        }
    }
    __syncwarp();   // the block is read before the buffer is reused as store staging
}

// Epilogue of 32 consecutive columns n0.. of one row.  coop: every lane of the
// warp holds a valid row (consecutive rows) and the 32 columns are in range, so
// the warp-cooperative loads / stores apply (all lanes take this path together).
// xa: this row's 32 aux values, already read from the chunk's TMA block (null: the
// aux matrix is read per thread here).
__device__ __forceinline__ void epilogue32(const TcParams& p, int b, int split, int row, int n0,
                                           float* v, uint8_t* stg, bool coop, const float* xa) {
    const int lane = threadIdx.x & 31;
    const bool full = n0 + 32 <= p.N;
    const int nv = full ? 32 : p.N - n0;
    if (p.ws) {
        const long i = ((long)(split * p.batch + b) * p.M + row) * p.N + n0;
        if (coop) wst32(stg, p.ws, i - (long)lane * p.N, p.N, NC_FP32, v);
        else if (full) st32(p.ws, i, NC_FP32, v);
        else {
#pragma unroll
            for (int j = 0; j < 32; ++j) if (j < nv) p.ws[i + j] = v[j];
        }
        return;
    }
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] *= p.alpha;
    const long ci = (long)b * p.sC + (long)row * p.ldc + n0;
    const long ai = (long)b * p.sAux + (long)row * p.ldaux + n0;
    if (p.epi == EPI_STORE) {
        const bool with_aux = p.aux && p.beta != 0.f;
        if (with_aux && xa) {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] += p.beta * xa[j];
        } else if (with_aux) {
            float a[32];
            if (full) ld32(p.aux, ai, p.aux_dtype, a);
            else {
#pragma unroll
                for (int j = 0; j < 32; ++j) a[j] = j < nv ? ld_elem(p.aux, ai + j, p.aux_dtype) : 0.f;
            }
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] += p.beta * a[j];
        }
        if (coop && (!with_aux || xa)) wst32(stg, p.C, ci - (long)lane * p.ldc, p.ldc, p.c_dtype, v);
        else if (full) st32(p.C, ci, p.c_dtype, v);
        else {
#pragma unroll
            for (int j = 0; j < 32; ++j) if (j < nv) st_elem(p.C, ci + j, p.c_dtype, v[j]);
        }
    } else if (p.epi == EPI_RELU2) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const float r = fmaxf(v[j], 0.f);
            v[j] = r * r;
        }
        if (coop) wst32(stg, p.C, ci - (long)lane * p.ldc, p.ldc, p.c_dtype, v);
        else if (full) st32(p.C, ci, p.c_dtype, v);
        else {
#pragma unroll
            for (int j = 0; j < 32; ++j) if (j < nv) st_elem(p.C, ci + j, p.c_dtype, v[j]);
        }
    } else {  // EPI_RELU2_BWD: dh = da * 2 relu(h) = da * 2 sqrt(a)
        // 2 relu(h) = 2 sqrt(a); a * rsqrt(a) (a > 0) is accurate far beyond bf16
        if (xa) {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] *= xa[j] > 0.f ? 2.f * xa[j] * rsqrtf(xa[j]) : 0.f;
        } else {
            float a[32];
            if (full) ld32(p.aux, ai, p.aux_dtype, a);
            else {
#pragma unroll
                for (int j = 0; j < 32; ++j) a[j] = j < nv ? ld_elem(p.aux, ai + j, p.aux_dtype) : 0.f;
            }
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] *= a[j] > 0.f ? 2.f * a[j] * rsqrtf(a[j]) : 0.f;
        }
        if (coop && xa) wst32(stg, p.C, ci - (long)lane * p.ldc, p.ldc, p.c_dtype, v);
        else if (full) st32(p.C, ci, p.c_dtype, v);
        else {
#pragma unroll
            for (int j = 0; j < 32; ++j) if (j < nv) st_elem(p.C, ci + j, p.c_dtype, v[j]);
        }
    }
}

// The epilogue of one accumulator tile for one row (this thread's TMEM lane),
// columns of group g (the first or second half of the tile).
// The transposed copy of a finished 32 x 32 chunk of a symmetric C: lane i holds
// row r0 + i, columns n0 .. n0+31 (final values); they are written to rows
// n0 .. n0+31, columns r0 .. r0+31.  coop: all 32 rows and columns are in range.
__device__ __forceinline__ void mirror32(const TcParams& p, uint8_t* stg, int b, int row, int n0, const float* v,
                                         bool coop) {
    const int lane = threadIdx.x & 31;
    const int r0 = row - lane;
    if (!coop) {
        if (row < p.M)
            for (int j = 0; j < 32 && n0 + j < p.N; ++j)
                st_elem(p.C, (long)b * p.sC + (long)(n0 + j) * p.ldc + row, p.c_dtype, v[j]);
        return;
    }
    float t[32];
    __syncwarp();
    if (p.c_dtype == NC_FP32) {
#pragma unroll
        for (int c = 0; c < 8; ++c)
            *reinterpret_cast<float4*>(stg + lane * 128 + ((c ^ (lane & 7)) << 4)) =
                make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
        __syncwarp();
#pragma unroll
        for (int r = 0; r < 32; ++r)
            t[r] = *reinterpret_cast<const float*>(stg + r * 128 + ((((lane >> 2) ^ (r & 7))) << 4) + (lane & 3) * 4);
    } else {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                __nv_bfloat162 h = __floats2bfloat162_rn(v[8 * c + 2 * e], v[8 * c + 2 * e + 1]);
                w[e] = *reinterpret_cast<uint32_t*>(&h);
            }
            *reinterpret_cast<uint4*>(stg + lane * 64 + ((c ^ ((lane >> 1) & 3)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
        }
        __syncwarp();
#pragma unroll
        for (int r = 0; r < 32; ++r)
            t[r] = __bfloat162float(*reinterpret_cast<const bf16*>(
                stg + r * 64 + ((((lane >> 3) ^ ((r >> 1) & 3))) << 4) + (lane & 7) * 2));
    }
    __syncwarp();
    wst32(stg, p.C, (long)b * p.sC + (long)n0 * p.ldc + r0, p.ldc, p.c_dtype, t);
}

// With p.aux_tma the blocks of the first x.slots chunks were issued by the caller;
// once a chunk is done, the block x.slots chunks ahead goes into its slot.
// Epilogue families a kernel instance is compiled for (each instance carries only its
// own epilogue code, which keeps the register budget of the others).
// The RMSNorm-backward pair: EF_DOT, the dh product that also leaves the row dots
// (EPI_RELU2_BWD with dot_out), and EF_NB, the dX product that finishes the norm (EPI_NORMB).
enum EpiFamily { EF_ANY = 0, EF_GEN = 1, EF_ROPE = 2, EF_DELTA = 3, EF_LSE = 4, EF_NB = 5, EF_DOT = 6 };
constexpr int epi_family(int epi, bool dot_out = false) {
    return epi == EPI_ROPE ? EF_ROPE : epi == EPI_DELTA ? EF_DELTA : epi == EPI_LSE ? EF_LSE
         : epi == EPI_NORMB ? EF_NB : (epi == EPI_RELU2_BWD && dot_out) ? EF_DOT : EF_GEN;
}

// MIRROR (compile time, symmetric products only): also write the transposed copy of
// each chunk when `mirror` (an off-diagonal tile).
template <int BN, bool MIRROR, int EF = EF_ANY>
__device__ __forceinline__ void epilogue_tile(const TcParams& p, int b, int split, int row, int tn,
                                              uint32_t tbase, int g, uint8_t* stg, XPipe& x,
                                              const CUtensorMap* mx, volatile int* abort, bool mirror,
                                              NextTile& nt) {
    const int lane = threadIdx.x & 31;
    const bool rows_ok = __all_sync(0xffffffffu, row < p.M);
    const int cend = (g + 1) * (BN / 64);
    if ((EF == EF_ANY || EF == EF_ROPE) && p.epi == EPI_ROPE) {
        // chunk pairs (a, a+2) hold head-dim pairs (j, j+64) of one 128-wide head; each
        // is done in two 16-column halves (bounded registers), staged for coalesced stores
        uint8_t* stg_b = stg + 2048;
#pragma unroll 1
        for (int pr = g * (BN / 128); pr < (g + 1) * (BN / 128); ++pr) {
            const int a = (pr >> 1) * 4 + (pr & 1);
            const int na = tn * BN + a * 32;
            const bool live = row < p.M && na < p.N;
            const long ci = (long)b * p.sC + (long)row * p.ldc + na;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                float va[16], vb[16];
                tc::tmem_ld16(tbase + a * 32 + 16 * hh, reinterpret_cast<uint32_t*>(va));
                tc::tmem_ld16(tbase + (a + 2) * 32 + 16 * hh, reinterpret_cast<uint32_t*>(vb));
                tc::tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    va[j] *= p.alpha;
                    vb[j] *= p.alpha;
                }
                if (live && na < p.rope_cols) {
                    // pair-major table: the warp's 32 rows (consecutive positions) read
                    // 256 contiguous bytes per pair
                    const float2* cs = p.rope + (long)((pr & 1) * 32 + 16 * hh) * p.rope_ld + (row % p.rope_T);
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const float2 c = __ldg(cs + (long)j * p.rope_ld);
                        const float x1 = va[j], x2 = vb[j];
                        va[j] = x1 * c.x - x2 * c.y;
                        vb[j] = x2 * c.x + x1 * c.y;
                    }
                }
                if (rows_ok) {
                    stage_bf16x16(stg, hh, va);
                    stage_bf16x16(stg_b, hh, vb);
                } else if (live) {
                    st16_bf16(reinterpret_cast<bf16*>(p.C) + ci + 16 * hh, va);
                    st16_bf16(reinterpret_cast<bf16*>(p.C) + ci + 64 + 16 * hh, vb);
                }
            }
            if (rows_ok && na < p.N) {
                flush_bf16(stg, p.C, ci - (long)lane * p.ldc, p.ldc);
                flush_bf16(stg_b, p.C, ci + 64 - (long)lane * p.ldc, p.ldc);
            }
        }
    } else if ((EF == EF_ANY || EF == EF_LSE) && p.epi == EPI_LSE) {
        // logits (bf16) out, and this row's (max, sum exp(z - max)) over the 128 columns of
        // this half of the tile, taken over the rounded values the cross-entropy will read
        constexpr float L2E = 1.4426950408889634f;
        float mx = -INFINITY, se = 0.f;
#pragma unroll 1
        for (int c = g * (BN / 64); c < (g + 1) * (BN / 64); ++c) {
            float v[32];
            tc::tmem_ld32(tbase + c * 32, reinterpret_cast<uint32_t*>(v));
            tc::tmem_wait_ld();
            const int n0 = tn * BN + c * 32;
            if (n0 < p.N) {   // warp-uniform
                float c4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
                uint32_t w[16];
#pragma unroll
                for (int j = 0; j < 32; j += 2) {
                    v[j] *= p.alpha;
                    v[j + 1] *= p.alpha;
                    w[j >> 1] = round_pack2(v[j], v[j + 1]);
                }
#pragma unroll
                for (int j = 0; j < 32; j += 2) c4[(j >> 1) & 3] = tc::fmax3(c4[(j >> 1) & 3], v[j], v[j + 1]);
                const float cm = fmaxf(fmaxf(c4[0], c4[1]), fmaxf(c4[2], c4[3]));
                if (cm > mx) {
                    se = mx == -INFINITY ? 0.f : se * tc::ex2a((mx - cm) * L2E);
                    mx = cm;
                }
                // sum of exp2(v * log2 e - mx * log2 e), two lanes at a time
                const uint64_t l2 = tc::f2pk(L2E, L2E), nml = tc::f2pk(-mx * L2E, -mx * L2E);
                uint64_t s2 = tc::f2pk(0.f, 0.f);
#pragma unroll
                for (int j = 0; j < 32; j += 2) {
                    float e0, e1;
                    tc::f2upk(tc::ffma2(tc::f2pk(v[j], v[j + 1]), l2, nml), e0, e1);
                    s2 = tc::fadd2(s2, tc::f2pk(tc::ex2a(e0), tc::ex2a(e1)));
                }
                {
                    float x0, x1;
                    tc::f2upk(s2, x0, x1);
                    se += x0 + x1;
                }
                const long ci = (long)b * p.sC + (long)row * p.ldc + n0;
                if (rows_ok) wst32_bf16w(stg, p.C, ci - (long)lane * p.ldc, p.ldc, w);
                else if (row < p.M) st32_bf16w(p.C, ci, w);
            }
        }
        const int grp = (tn * BN + g * (BN / 2)) / 128;
        if (row < p.M && grp * 128 < p.N) p.lse_part[(long)row * (p.N / 128) + grp] = make_float2(mx, se);
    } else if ((EF == EF_ANY || EF == EF_DELTA) && p.epi == EPI_DELTA) {
        // dO (bf16) out; per 128-column head the dot product with O (aux) of the
        // rounded values, i.e. exactly what the attention backward will consume
        float dot = 0.f;
#pragma unroll 1
        for (int c = g * (BN / 64); c < (g + 1) * (BN / 64); ++c) {
            float v[32];
            tc::tmem_ld32(tbase + c * 32, reinterpret_cast<uint32_t*>(v));
            tc::tmem_wait_ld();
            const int n0 = tn * BN + c * 32;
            const uint8_t* xb = nullptr;
            float o[32];
            if (p.aux_tma) {
                if (!(xb = x_wait(x, abort))) break;
                x_row(xb, NC_BF16, o);
            }
            if (row < p.M && n0 < p.N) {
                uint32_t w[16];
#pragma unroll
                for (int j = 0; j < 32; j += 2) {
                    v[j] *= p.alpha;
                    v[j + 1] *= p.alpha;
                    w[j >> 1] = round_pack2(v[j], v[j + 1]);
                }
                const long ci = (long)b * p.sC + (long)row * p.ldc + n0;
                const long ai = (long)b * p.sAux + (long)row * p.ldaux + n0;
                {
                    if (!xb) ld32(p.aux, ai, NC_BF16, o);
#pragma unroll
                    for (int j = 0; j < 32; ++j) dot = fmaf(v[j], o[j], dot);
                    if (xb && rows_ok) wst32_bf16w(const_cast<uint8_t*>(xb), p.C, ci - (long)lane * p.ldc, p.ldc, w);
                    else st32_bf16w(p.C, ci, w);
                }
                if ((c & 3) == 3) {
                    const int hh = n0 / 128, t = row % p.rope_T, bb = row / p.rope_T;
                    p.delta[((long)bb * (p.N / 128) + hh) * p.rope_T + t] = dot;
                    dot = 0.f;
                }
            }
            if (p.aux_tma) x_ahead(x, mx, g * (BN / 64), cend, BN, tn, row, b, nt);
        }
    } else if (EF == EF_NB) {
        // RMSNorm backward, dy = alpha acc never stored: this row's D = <dy, y> from the
        // partials its producers left, then per chunk g = gin + r (dy - y D / d) in fp32
        // and its bf16 copy.  N is a multiple of 128, so a chunk is whole or absent.  The
        // residual gradient in (fp32, read per lane) is fetched one chunk ahead.
        const bool live = row < p.M;
        float rr = 0.f, dm = 0.f;
        if (live) {
            rr = p.nb_r[row];
            const float* pp = p.nb_part + (long)row * p.nb_nparts;
            float sd = 0.f;
            if ((p.nb_nparts & 3) == 0) {
#pragma unroll 4
                for (int k = 0; k < p.nb_nparts; k += 4) {
                    const float4 f = *reinterpret_cast<const float4*>(pp + k);
                    sd = (((sd + f.x) + f.y) + f.z) + f.w;
                }
            } else {
                for (int k = 0; k < p.nb_nparts; ++k) sd += pp[k];
            }
            dm = sd * p.nb_inv_d;
        }
        float* C = reinterpret_cast<float*>(p.C);
        const int cstart = g * (BN / 64);
        float gi[32];
        auto fetch_gin = [&](int c) {
            const int n0 = tn * BN + c * 32;
            if (p.nb_gin && live && n0 < p.N) ld32(p.nb_gin, (long)row * p.ldc + n0, NC_FP32, gi);
            else {
#pragma unroll
                for (int j = 0; j < 32; ++j) gi[j] = 0.f;
            }
        };
        fetch_gin(cstart);
#pragma unroll 1
        for (int c = cstart; c < cend; ++c) {
            float v[32];
            tc::tmem_ld32(tbase + c * 32, reinterpret_cast<uint32_t*>(v));
            tc::tmem_wait_ld();
            const int n0 = tn * BN + c * 32;
            const uint8_t* xb = nullptr;
            {
                float y[32];
                if (p.aux_tma) {
                    if (!(xb = x_wait(x, abort))) break;
                    x_row(xb, NC_BF16, y);
                } else if (live && n0 < p.N) {
                    ld32(p.aux, (long)row * p.ldaux + n0, NC_BF16, y);
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) y[j] = 0.f;
                }
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = gi[j] + rr * (p.alpha * v[j] - y[j] * dm);
            }
            if (c + 1 < cend) fetch_gin(c + 1);
            if (n0 < p.N) {   // warp-uniform
                const long ci = (long)row * p.ldc + n0;
                if (rows_ok) {
                    uint8_t* sb = xb ? const_cast<uint8_t*>(xb) : stg;
                    const long c0 = ci - (long)lane * p.ldc;
                    wst16_f32(sb, C, c0, p.ldc, v);
                    wst16_f32(sb, C, c0 + 16, p.ldc, v + 16);
                    wst32(sb, p.nb_gt, c0, p.ldc, NC_BF16, v);
                } else if (live) {
                    st32(C, ci, NC_FP32, v);
                    st32(p.nb_gt, ci, NC_BF16, v);
                }
            }
            if (p.aux_tma) x_ahead(x, mx, g * (BN / 64), cend, BN, tn, row, b, nt);
        }
    } else if (EF == EF_DOT) {
        // dh = alpha acc * 2 relu(h) = alpha acc * 2 sqrt(a), and per 128-column group the
        // row dot <dh, relu(h)> over the stored (rounded) dh: the dot product <dy, y> the
        // RMSNorm backward after the next product needs (dy = dh W1, h = W1 y)
        float dot = 0.f;
#pragma unroll 1
        for (int c = g * (BN / 64); c < cend; ++c) {
            float v[32];
            tc::tmem_ld32(tbase + c * 32, reinterpret_cast<uint32_t*>(v));
            tc::tmem_wait_ld();
            const int n0 = tn * BN + c * 32;
            const uint8_t* xb = nullptr;
            float a[32];
            if (p.aux_tma) {
                if (!(xb = x_wait(x, abort))) break;
                x_row(xb, NC_BF16, a);
            }
            if (n0 < p.N) {   // warp-uniform
                const long ci = (long)row * p.ldc + n0;
                if (!xb && row < p.M) ld32(p.aux, (long)row * p.ldaux + n0, NC_BF16, a);
                uint32_t w[16];
#pragma unroll
                for (int j = 0; j < 32; j += 2) {
                    const float s0 = a[j] > 0.f ? a[j] * rsqrtf(a[j]) : 0.f;
                    const float s1 = a[j + 1] > 0.f ? a[j + 1] * rsqrtf(a[j + 1]) : 0.f;
                    float x0 = v[j] * p.alpha * (2.f * s0), x1 = v[j + 1] * p.alpha * (2.f * s1);
                    w[j >> 1] = round_pack2(x0, x1);
                    dot = fmaf(x0, s0, dot);
                    dot = fmaf(x1, s1, dot);
                }
                if (rows_ok) wst32_bf16w(xb ? const_cast<uint8_t*>(xb) : stg, p.C, ci - (long)lane * p.ldc, p.ldc, w);
                else if (row < p.M) st32_bf16w(p.C, ci, w);
            }
            if (p.aux_tma) x_ahead(x, mx, g * (BN / 64), cend, BN, tn, row, b, nt);
        }
        const int grp = (tn * BN + g * (BN / 2)) / 128;
        if (row < p.M && grp * 128 < p.N) p.dot_out[(long)row * (p.N / 128) + grp] = dot;
    } else if (EF != EF_NB && EF != EF_DOT)
#pragma unroll 1
    for (int c = g * (BN / 64); c < (g + 1) * (BN / 64); ++c) {
        float v[32];
        tc::tmem_ld32(tbase + c * 32, reinterpret_cast<uint32_t*>(v));
        tc::tmem_wait_ld();
        const int n0 = tn * BN + c * 32;
        const uint8_t* xb = nullptr;
        float a[32];
        if (p.aux_tma) {
            if (!(xb = x_wait(x, abort))) break;
            x_row(xb, p.aux_dtype, a);
        }
        if (row < p.M && n0 < p.N) {
            epilogue32(p, b, split, row, n0, v, xb ? const_cast<uint8_t*>(xb) : stg,
                       rows_ok && n0 + 32 <= p.N, xb ? a : nullptr);
        }
        if constexpr (MIRROR) {
            if (mirror && n0 < p.N)   // symmetric C: the transposed copy of this chunk (warp-uniform)
                mirror32(p, xb ? const_cast<uint8_t*>(xb) : stg, b, row, n0, v, rows_ok && n0 + 32 <= p.N);
        }
        if (p.aux_tma) x_ahead(x, mx, g * (BN / 64), cend, BN, tn, row, b, nt);
    }
}

template <int BN, bool A_MN, bool B_MN>
__global__ void __launch_bounds__(NTHREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmX, const TcParams p) {
    using C = Cfg<BN>;
    constexpr int S = C::STAGES;
    constexpr uint32_t IDESC = tc::idesc_bf16(BM, BN, A_MN, B_MN);
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t* epi_smem = smem + S * C::STAGE;   // 1024-aligned: the swizzled TMA blocks need it
    uint64_t* full = reinterpret_cast<uint64_t*>(epi_smem + EPI_STG_BYTES);
    uint64_t* empty = full + S;
    uint64_t* tfull = empty + S;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint64_t* xbar = drain + 1;   // [EPI_WARPS][XSLOTS_MAX]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(xbar + XSLOTS_MAX * EPI_WARPS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            tc::mbar_init(&full[s], 1);
            tc::mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            tc::mbar_init(&tfull[a], 1);
            tc::mbar_init(&tempty[a], EPI_WARPS * 32);
        }
        tc::mbar_init(drain, 1);
        for (int i = 0; i < XSLOTS_MAX * EPI_WARPS; ++i) tc::mbar_init(&xbar[i], 1);
        *abort_flag = 0;
        tc::fence_barrier_init();
        tc::tma_prefetch(&tmA);
        tc::tma_prefetch(&tmB);
        if (p.aux_tma) tc::tma_prefetch(&tmX);
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, C::TMEM_COLS);
        tc::tmem_relinquish();
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0 && lane == 0) {
        // ---------------------------------------------------- TMA producer
        int stage = 0;
        uint32_t ph = 0;
        long issued = 0;
        for (long u = blockIdx.x; u < p.units; u += gridDim.x) {
            int b, split, tm, tn, kb0, kb1;
            decode(p, u, b, split, tm, tn);
            kb_range(p, split, kb0, kb1);
            bool ok = true;
            for (int kb = kb0; kb < kb1; ++kb) {
                if (!tc::mbar_wait(&empty[stage], ph ^ 1, abort_flag)) { ok = false; break; }
                uint8_t* sa = smem + stage * C::STAGE;
                uint8_t* sb = sa + C::A_BYTES;
                tc::mbar_expect_tx(&full[stage], C::STAGE);
                if (!A_MN) {
                    tc::tma_load_3d(sa, &tmA, &full[stage], kb * BK, tm * BM, b);
                } else {
                    tc::tma_load_3d(sa, &tmA, &full[stage], tm * BM, kb * BK, b);
                    tc::tma_load_3d(sa + 8192, &tmA, &full[stage], tm * BM + 64, kb * BK, b);
                }
                if (!B_MN) {
                    tc::tma_load_3d(sb, &tmB, &full[stage], kb * BK, tn * BN, b);
                } else {
#pragma unroll
                    for (int j = 0; j < BN / 64; ++j)
                        tc::tma_load_3d(sb + j * 8192, &tmB, &full[stage], tn * BN + j * 64, kb * BK, b);
                }
                ++issued;
                if (++stage == S) { stage = 0; ph ^= 1; }
            }
            if (!ok) break;
        }
        if (*abort_flag) {
            // let the copies still in flight land before the CTA exits
            int st = stage;
            uint32_t sp = ph;
            for (long i = 0; i < issued && i < S; ++i) {
                if (st == 0) { st = S - 1; sp ^= 1; } else { --st; }
                tc::mbar_wait_drain(&full[st], sp);
            }
        }
    } else if (warp == 1 && lane == 0) {
        // ---------------------------------------------------- MMA issuer
        int stage = 0, acc = 0;
        uint32_t ph = 0, aph = 0;
        for (long u = blockIdx.x; u < p.units; u += gridDim.x) {
            int b, split, tm, tn, kb0, kb1;
            decode(p, u, b, split, tm, tn);
            kb_range(p, split, kb0, kb1);
            if (!tc::mbar_wait(&tempty[acc], aph ^ 1, abort_flag)) break;
            tc::fence_after();
            const uint32_t d = tmem + (uint32_t)(acc * BN);
            bool ok = true;
            for (int kb = kb0; kb < kb1; ++kb) {
                if (!tc::mbar_wait(&full[stage], ph, abort_flag)) { ok = false; break; }
                tc::fence_after();
                const uint32_t a0 = tc::smem_u32(smem + stage * C::STAGE);
                const uint32_t b0 = a0 + C::A_BYTES;
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk) {
                    const uint64_t ad = A_MN ? tc::sdesc(a0 + kk * 2048, 8192, 1024)
                                             : tc::sdesc(a0 + kk * 32, 16, 1024);
                    const uint64_t bd = B_MN ? tc::sdesc(b0 + kk * 2048, 8192, 1024)
                                             : tc::sdesc(b0 + kk * 32, 16, 1024);
                    tc::mma_bf16(d, ad, bd, IDESC, (kb > kb0 || kk > 0) ? 1u : 0u);
                }
                tc::mma_commit(&empty[stage]);
                if (++stage == S) { stage = 0; ph ^= 1; }
            }
            if (!ok) break;
            tc::mma_commit(&tfull[acc]);
            acc ^= 1;
            if (acc == 0) aph ^= 1;
        }
        if (*abort_flag) {
            tc::mma_commit(drain);
            tc::mbar_wait_drain(drain, 0);
        }
    } else if (warp >= 2) {
        // ---------------------------------------------------- epilogue
        const int q = warp & 3, g = (warp - 2) >> 2;
        const bool xf32 = p.aux_dtype == NC_FP32;
        XPipe x = x_make(epi_smem + (warp - 2) * EPI_STG, xbar + XSLOTS_MAX * (warp - 2), xf32);
        int acc = 0;
        uint32_t aph = 0;
        int carried = 0;   // aux blocks of this tile fetched during the last epilogue
        for (long u = blockIdx.x; u < p.units; u += gridDim.x) {
            int b, split, tm, tn;
            decode(p, u, b, split, tm, tn);
            const int row = tm * BM + q * 32 + lane;
            NextTile nt{false, 0, 0, 0, 0};
            if (p.aux_tma && u + gridDim.x < p.units) {
                int s2, tm2;
                decode(p, u + gridDim.x, nt.b, s2, tm2, nt.tn);
                nt.row = tm2 * BM + q * 32 + lane;
                nt.on = true;
            }
            if (p.aux_tma) {   // this tile's first blocks come in while its MMAs run
                const int first = min(x.slots(), BN / 64);
                for (int k = carried; k < first; ++k) x_issue(x, &tmX, tn * BN + g * (BN / 2) + 32 * k, row - lane, b);
                nt.next = max(carried, first);
            }
            if (!tc::mbar_wait_warp(&tfull[acc], aph, abort_flag)) break;
            tc::fence_after();
            const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
            epilogue_tile<BN, false>(p, b, split, row, tn, tbase, g, x.bufp(0), x, &tmX, abort_flag, false, nt);
            carried = max(0, nt.next - BN / 64);
            tc::fence_before();
            tc::mbar_arrive(&tempty[acc]);
            acc ^= 1;
            if (acc == 0) aph ^= 1;
        }
        if (*abort_flag) x_drain(x);
    }

    tc::fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && *abort_flag && p.flag) atomicOr(p.flag, NC_FLAG_TIMEOUT);
    if (warp == 1) {
        tc::fence_after();
        tc::tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

// ---------------------------------------------------------------- CTA-pair kernel
// Two CTAs of a cluster share one 256 x 256 output tile: CTA rank r owns rows
// [128 r, 128 r + 128) of A and of B (the N rows), and its TMEM holds its 128
// output rows.  The leader (rank 0) issues tcgen05.mma.cta_group::2 (M=256,
// N=256, K=16), which reads A and B halves from both CTAs' shared memory, so
// each SM streams half the operand bytes per FLOP of the 1-CTA tile.  Both
// CTAs' TMA loads complete on the leader's full barrier; the leader's commits
// multicast to both CTAs' empty / accumulator-full barriers; both CTAs'
// epilogue warps release an accumulator on the leader's barrier.
constexpr int P_BN = 256, P_STAGES = 5;
constexpr int P_A_BYTES = 128 * BK * 2, P_B_BYTES = 128 * BK * 2;
constexpr int P_STAGE = P_A_BYTES + P_B_BYTES;
constexpr int P_SMEM = P_STAGES * P_STAGE + 1024 + BAR_BYTES + EPI_STG_BYTES;

template <bool A_MN, bool B_MN, bool SYM, int EF>
__global__ void __launch_bounds__(NTHREADS, 1)
    gemm_tc2_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmX, const TcParams p) {
    constexpr int S = P_STAGES;
    constexpr uint32_t IDESC = tc::idesc_bf16(256, P_BN, A_MN, B_MN);
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t* epi_smem = smem + S * P_STAGE;   // 1024-aligned: the swizzled TMA blocks need it
    uint64_t* full = reinterpret_cast<uint64_t*>(epi_smem + EPI_STG_BYTES);
    uint64_t* empty = full + S;
    uint64_t* tfull = empty + S;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint64_t* xbar = drain + 1;   // [EPI_WARPS][XSLOTS_MAX]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(xbar + XSLOTS_MAX * EPI_WARPS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t rank = tc::cluster_ctarank();
    const long cluster = blockIdx.x >> 1, nclusters = gridDim.x >> 1;
    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            tc::mbar_init(&full[i], 1);
            tc::mbar_init(&empty[i], 1);
        }
        for (int a = 0; a < 2; ++a) {
            tc::mbar_init(&tfull[a], 1);
            tc::mbar_init(&tempty[a], 2 * EPI_WARPS);   // every epilogue warp of both CTAs
        }
        tc::mbar_init(drain, 1);
        for (int i = 0; i < XSLOTS_MAX * EPI_WARPS; ++i) tc::mbar_init(&xbar[i], 1);
        *abort_flag = 0;
        tc::fence_barrier_init();
        tc::tma_prefetch(&tmA);
        tc::tma_prefetch(&tmB);
        if (p.aux_tma) tc::tma_prefetch(&tmX);
    }
    if (warp == 1) {
        tc::tmem_alloc2(tmem_slot, 512);
        tc::tmem_relinquish2();
    }
    tc::fence_before();
    __syncthreads();
    tc::cluster_sync();   // barriers of both CTAs initialised before any cross-CTA signal
    tc::fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0 && lane == 0) {
        // ---------------------------------------------------- TMA producer (both CTAs)
        int stage = 0;
        uint32_t ph = 0;
        for (long u = cluster; u < p.units; u += nclusters) {
            int b, split, tm, tn, kb0, kb1;
            decode(p, u, b, split, tm, tn);
            kb_range(p, split, kb0, kb1);
            const int row_a = tm * 256 + (int)rank * 128, row_b = tn * P_BN + (int)rank * 128;
            bool ok = true;
            for (int kb = kb0; kb < kb1; ++kb) {
                if (!tc::mbar_wait(&empty[stage], ph ^ 1, abort_flag)) { ok = false; break; }
                uint8_t* sa = smem + stage * P_STAGE;
                uint8_t* sb = sa + P_A_BYTES;
                const uint32_t fb = tc::mapa(tc::smem_u32(&full[stage]), 0);
                if (rank == 0) tc::mbar_expect_tx(&full[stage], 2 * P_STAGE);
                if (!A_MN) {
                    tc::tma_load_3d_pair(sa, &tmA, fb, kb * BK, row_a, b);
                } else {
                    tc::tma_load_3d_pair(sa, &tmA, fb, row_a, kb * BK, b);
                    tc::tma_load_3d_pair(sa + 8192, &tmA, fb, row_a + 64, kb * BK, b);
                }
                if (!B_MN) {
                    tc::tma_load_3d_pair(sb, &tmB, fb, kb * BK, row_b, b);
                } else {
                    tc::tma_load_3d_pair(sb, &tmB, fb, row_b, kb * BK, b);
                    tc::tma_load_3d_pair(sb + 8192, &tmB, fb, row_b + 64, kb * BK, b);
                }
                if (++stage == S) { stage = 0; ph ^= 1; }
            }
            if (!ok) break;
        }
    } else if (warp == 1 && lane == 0 && rank == 0) {
        // ---------------------------------------------------- MMA issuer (leader only)
        int stage = 0, acc = 0;
        uint32_t ph = 0, aph = 0;
        for (long u = cluster; u < p.units; u += nclusters) {
            int b, split, tm, tn, kb0, kb1;
            decode(p, u, b, split, tm, tn);
            kb_range(p, split, kb0, kb1);
            if (!tc::mbar_wait(&tempty[acc], aph ^ 1, abort_flag)) break;
            tc::fence_after();
            const uint32_t d = tmem + (uint32_t)(acc * P_BN);
            bool ok = true;
            for (int kb = kb0; kb < kb1; ++kb) {
                if (!tc::mbar_wait(&full[stage], ph, abort_flag)) { ok = false; break; }
                tc::fence_after();
                const uint32_t a0 = tc::smem_u32(smem + stage * P_STAGE);
                const uint32_t b0 = a0 + P_A_BYTES;
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk) {
                    const uint64_t ad = A_MN ? tc::sdesc(a0 + kk * 2048, 8192, 1024)
                                             : tc::sdesc(a0 + kk * 32, 16, 1024);
                    const uint64_t bd = B_MN ? tc::sdesc(b0 + kk * 2048, 8192, 1024)
                                             : tc::sdesc(b0 + kk * 32, 16, 1024);
                    tc::mma2_bf16(d, ad, bd, IDESC, (kb > kb0 || kk > 0) ? 1u : 0u);
                }
                tc::mma2_commit_mc(&empty[stage], 0x3);
                if (++stage == S) { stage = 0; ph ^= 1; }
            }
            if (!ok) break;
            tc::mma2_commit_mc(&tfull[acc], 0x3);
            acc ^= 1;
            if (acc == 0) aph ^= 1;
        }
        if (*abort_flag) {
            tc::mma2_commit_mc(drain, 0x1);
            tc::mbar_wait_drain(drain, 0);
        }
    } else if (warp >= 2) {
        // ---------------------------------------------------- epilogue (both CTAs)
        const int q = warp & 3, g = (warp - 2) >> 2;
        const bool xf32 = p.aux_dtype == NC_FP32;
        XPipe x = x_make(epi_smem + (warp - 2) * EPI_STG, xbar + XSLOTS_MAX * (warp - 2), xf32);
        const uint32_t tempty_leader = tc::mapa(tc::smem_u32(&tempty[0]), 0);
        int acc = 0;
        uint32_t aph = 0;
        int carried = 0;   // aux blocks of this tile fetched during the last epilogue
        for (long u = cluster; u < p.units; u += nclusters) {
            int b, split, tm, tn;
            decode(p, u, b, split, tm, tn);
            const int row = tm * 256 + (int)rank * 128 + q * 32 + lane;
            NextTile nt{false, 0, 0, 0, 0};
            if (p.aux_tma && u + nclusters < p.units) {
                int s2, tm2;
                decode(p, u + nclusters, nt.b, s2, tm2, nt.tn);
                nt.row = tm2 * 256 + (int)rank * 128 + q * 32 + lane;
                nt.on = true;
            }
            if (p.aux_tma) {   // this tile's first blocks come in while its MMAs run
                const int first = min(x.slots(), P_BN / 64);
                for (int k = carried; k < first; ++k)
                    x_issue(x, &tmX, tn * P_BN + g * (P_BN / 2) + 32 * k, row - lane, b);
                nt.next = max(carried, first);
            }
            if (!tc::mbar_wait_warp(&tfull[acc], aph, abort_flag)) break;
            tc::fence_after();
            const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * P_BN);
            epilogue_tile<P_BN, SYM, EF>(p, b, split, row, tn, tbase, g, x.bufp(0), x, &tmX, abort_flag,
                                     SYM && tm != tn, nt);
            carried = max(0, nt.next - P_BN / 64);
            tc::fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive_cluster(tempty_leader + acc * 8);
            acc ^= 1;
            if (acc == 0) aph ^= 1;
        }
        if (*abort_flag) x_drain(x);
    }

    tc::fence_before();
    __syncthreads();
    tc::cluster_sync();   // no CTA leaves while its peer may still signal it
    if (threadIdx.x == 0 && *abort_flag && p.flag) atomicOr(p.flag, NC_FLAG_TIMEOUT);
    if (warp == 1) {
        tc::fence_after();
        tc::tmem_dealloc2(tmem, 512);
    }
}

// C = alpha * sum_s ws[s] + beta * aux, fixed summation order.
__device__ __forceinline__ float split_epi(float v, int epi) {
    if (epi == EPI_RELU2) {
        const float r = fmaxf(v, 0.f);
        return r * r;
    }
    return v;
}

__global__ void splitk_reduce_kernel(const float* ws, int splits, int batch, int M, int N, void* C,
                                     long ldc, long sC, int c_dtype, const void* aux, long ldaux,
                                     long sAux, int aux_dtype, float alpha, float beta, int epi) {
    const long total = (long)batch * M * N;
    const long i = (long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= total) return;
    const long n = i % N, m = (i / N) % M, b = i / ((long)N * M);
    float s = 0.f;
    for (int k = 0; k < splits; ++k) s += ws[(long)k * total + i];
    s *= alpha;
    if (epi == EPI_STORE && aux && beta != 0.f) s += beta * ld_elem(aux, b * sAux + m * ldaux + n, aux_dtype);
    st_elem(C, b * sC + m * ldc + n, c_dtype, split_epi(s, epi));
}

// The same, four consecutive columns per thread (16-byte loads of every partial) and 32-bit
// index arithmetic; needs N, ldc, ldaux multiples of 4, 16-byte aligned bases and fewer
// than 2^31 quads.
__global__ void __launch_bounds__(256) splitk_reduce4_kernel(const float* ws, int splits, int rows, int M,
                                                             int N, void* C, long ldc, long sC, int c_dtype,
                                                             const void* aux, long ldaux, long sAux,
                                                             int aux_dtype, float alpha, float beta,
                                                             int epi) {
    const int n4 = N / 4;
    const long total = (long)rows * N;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < rows * n4; i += gridDim.x * blockDim.x) {
        const int r = i / n4, c = (i - r * n4) * 4;
        const int b = r / M, m = r - b * M;
        const long wi = (long)r * N + c;
        float4 acc = reinterpret_cast<const float4*>(ws + wi)[0];
        for (int k = 1; k < splits; ++k) {
            const float4 v = reinterpret_cast<const float4*>(ws + (long)k * total + wi)[0];
            acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
        }
        float o[4] = {acc.x * alpha, acc.y * alpha, acc.z * alpha, acc.w * alpha};
        if (epi == EPI_STORE && aux && beta != 0.f) {
            const long ai = (long)b * sAux + (long)m * ldaux + c;
            if (aux_dtype == NC_FP32) {
                const float4 a = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(aux) + ai)[0];
                o[0] += beta * a.x; o[1] += beta * a.y; o[2] += beta * a.z; o[3] += beta * a.w;
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e) o[e] += beta * ld_elem(aux, ai + e, aux_dtype);
            }
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) o[e] = split_epi(o[e], epi);
        const long ci = (long)b * sC + (long)m * ldc + c;
        if (c_dtype == NC_FP32) {
            reinterpret_cast<float4*>(reinterpret_cast<float*>(C) + ci)[0] = make_float4(o[0], o[1], o[2], o[3]);
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) st_elem(C, ci + e, c_dtype, o[e]);
        }
    }
}

template <int BN, bool A_MN, bool B_MN>
int launch(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& mx, const TcParams& p,
           cudaStream_t s) {
    using C = Cfg<BN>;
    static DeviceOnce attr;
    NC_TRY(attr.run([] {
        return cuda_check(cudaFuncSetAttribute(gemm_tc_kernel<BN, A_MN, B_MN>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM),
                          "gemm_tc smem attribute");
    }));
    const long grid = p.units < num_sms() ? p.units : num_sms();
    gemm_tc_kernel<BN, A_MN, B_MN><<<(int)grid, NTHREADS, C::SMEM, s>>>(ma, mb, mx, p);
    note_launch();
    NC_LAUNCH_CHECK("gemm_tc");
    return NC_OK;
}

template <bool A_MN, bool B_MN, bool SYM = false, int EF = EF_GEN>
int launch2(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& mx, const TcParams& p,
            cudaStream_t s) {
    static DeviceOnce attr;
    NC_TRY(attr.run([] {
        return cuda_check(cudaFuncSetAttribute(gemm_tc2_kernel<A_MN, B_MN, SYM, EF>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, P_SMEM),
                          "gemm_tc2 smem attribute");
    }));
    long clusters = p.units < num_sms() / 2 ? p.units : num_sms() / 2;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(2 * clusters), 1, 1);
    cfg.blockDim = dim3(NTHREADS, 1, 1);
    cfg.dynamicSmemBytes = P_SMEM;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    NC_TRY(cuda_check(cudaLaunchKernelEx(&cfg, gemm_tc2_kernel<A_MN, B_MN, SYM, EF>, ma, mb, mx, p), "gemm_tc2 launch"));
    note_launch();
    NC_LAUNCH_CHECK("gemm_tc2");
    return NC_OK;
}

// Fraction of the slots busy when `units` work items run in waves of `slots`.
double wave_eff(long units, int slots) {
    const long waves = (units + slots - 1) / slots;
    return (double)units / ((double)waves * slots);
}

// Split K over CTAs when that fills the GPU's waves better.  Modelled time: the
// larger of the MMA work at ~1.4 PFLOP/s divided by the wave efficiency and the
// operand bytes at ~50 GB/s per CTA (at most ~6 TB/s), plus, for s > 1, writing
// and re-reading s fp32 partials of the output at ~6 TB/s.  This splits the
// long-K, small-output weight gradients and, where the operand stream is the
// bound (a few token rows against a weight matrix), the small-N products.
int pick_splits(const Gemm& g, int tiles, int num_kb, int slots) {
    if ((g.epi != EPI_STORE && g.epi != EPI_RELU2) || num_kb < 8) return 1;
    const long work = (long)tiles * g.batch;
    const double flops = 2.0 * g.M * g.N * (double)g.K * g.batch;
    const double op_bytes = ((double)g.M + g.N) * g.K * g.batch * 2.0;
    const double out_bytes = (double)g.M * g.N * g.batch * 4.0;
    auto cost = [&](int s) {
        const double mma = flops / 1.4e15 / wave_eff(work * s, slots);
        const double mem = op_bytes / fmin(6.0e12, (double)fmin(work * s, (long)slots) * 5.0e10);
        return fmax(mma, mem) + (s > 1 ? 2.0 * s * out_bytes / 6.0e12 : 0.0);
    };
    const bool mem_bound = op_bytes / 6.0e12 > flops / 1.4e15;
    const int min_kb = mem_bound ? 4 : 8;
    if (num_kb < 2 * min_kb) return 1;
    int bs = 1;
    double best = cost(1);
    for (int s = 2; s <= 16 && num_kb / s >= min_kb; ++s) {
        const double c = cost(s);
        if (c < 0.97 * best) {
            best = c;
            bs = s;
        }
    }
    return bs;
}

}  // namespace

// ------------------------------------------------------------ host side (shared with attention)
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// 3-D bf16 tensor map over [batch][outer][inner] (row stride ld, batch stride bs, in elements).
int make_map(CUtensorMap* m, const void* ptr, long inner, long outer, long batch, long ld, long bs,
             int box_inner, int box_outer) {
    auto fn = encode_fn();
    if (!fn) return set_error(NC_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
    if (batch <= 1) bs = ld * outer;
    cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)outer, (cuuint64_t)(batch < 1 ? 1 : batch)};
    cuuint64_t strides[2] = {(cuuint64_t)ld * 2, (cuuint64_t)bs * 2};
    cuuint32_t box[3] = {(cuuint32_t)box_inner, (cuuint32_t)box_outer, 1};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box,
                    es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return set_error(NC_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d): inner %ld outer %ld ld %ld",
                         (int)r, inner, outer, ld);
    return NC_OK;
}

// 3-D map of an fp32 / bf16 matrix [batch][outer][inner] for the epilogue's 32 x 32
// blocks, swizzled so that row r's 16-byte chunk c lands at chunk c ^ (r & 7) (fp32,
// 128-byte rows) or c ^ ((r >> 1) & 3) (bf16, 64-byte rows).
int make_map_x(CUtensorMap* m, const void* ptr, int dt, long inner, long outer, long batch, long ld, long bs) {
    auto fn = encode_fn();
    if (!fn) return set_error(NC_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
    const int es = dt == NC_FP32 ? 4 : 2;
    if (batch <= 1) bs = ld * outer;
    cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)outer, (cuuint64_t)(batch < 1 ? 1 : batch)};
    cuuint64_t strides[2] = {(cuuint64_t)ld * es, (cuuint64_t)bs * es};
    cuuint32_t box[3] = {32, 32, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, dt == NC_FP32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                    const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    dt == NC_FP32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return set_error(NC_ERR_CUDA, "cuTensorMapEncodeTiled (aux) failed (%d): inner %ld outer %ld ld %ld",
                         (int)r, inner, outer, ld);
    return NC_OK;
}

int num_sms() {
    static int n = 0;
    if (!n) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (n <= 0) n = 148;
    }
    return n;
}


bool gemm_tc_supported(const Gemm& g) {
    if (g.in_dtype != NC_BF16) return false;
    if (g.M <= 0 || g.N <= 0 || g.K <= 0) return false;
    if (g.lda % 8 || g.ldb % 8 || g.ldc % 8 || (g.aux && g.ldaux % 8)) return false;
    if (g.batch > 1 && (g.sA % 8 || g.sB % 8)) return false;
    if ((uintptr_t)g.A % 16 || (uintptr_t)g.B % 16 || (uintptr_t)g.C % 16) return false;
    if (g.aux && (uintptr_t)g.aux % 16) return false;
    if (g.N % 8) return false;
    if (g.epi == EPI_ROPE && (g.N % 128 || !g.rope || g.rope_T <= 0 || g.rope_ld < g.rope_T ||
                              g.c_dtype != NC_BF16)) return false;
    if (g.epi == EPI_LSE && (g.N % 128 || g.N < 256 || !g.lse_part || g.c_dtype != NC_BF16 || g.batch != 1))
        return false;
    // the CTA-pair instances of the special epilogues exist for the layouts the step uses
    if ((g.epi == EPI_ROPE || g.epi == EPI_LSE) && (g.a_t || g.b_t)) return false;
    if (g.epi == EPI_DELTA && (g.a_t || !g.b_t)) return false;
    if (g.epi == EPI_DELTA && (g.N % 128 || g.N < 256 || !g.delta || !g.aux || g.rope_T <= 0 || g.c_dtype != NC_BF16 ||
                               g.aux_dtype != NC_BF16 || g.batch != 1))
        return false;
    // the RMSNorm-backward pair: CTA-pair tiles (two 128-column groups per tile), A K-major,
    // B MN-major (the dX and dh products of the backward), one matrix
    const bool nb_shape = g.M >= 256 && g.N >= 256 && g.N % 128 == 0 && !g.a_t && g.b_t && g.batch == 1;
    if (g.dot_out && (g.epi != EPI_RELU2_BWD || !nb_shape || !g.aux || g.aux_dtype != NC_BF16 ||
                      g.c_dtype != NC_BF16))
        return false;
    if (g.epi == EPI_NORMB &&
        (!nb_shape || !g.aux || g.aux_dtype != NC_BF16 || g.c_dtype != NC_FP32 || !g.nb_r || !g.nb_part ||
         g.nb_nparts <= 0 || !g.nb_gt || (uintptr_t)g.nb_gt % 16 || (uintptr_t)g.nb_gin % 16))
        return false;
    return true;
}

// CTA pairs (256 x 256 tiles) for every GEMM big enough to fill them.
static bool use_pairs(const Gemm& g) { return g.M >= 256 && g.N >= 256; }

double gemm_tc_work_fraction(const Gemm& g) {
    if (!(g.sym && use_pairs(g) && g.M == g.N && g.epi == EPI_STORE && !g.a_t)) return 1.0;
    const double t = ceil_div(g.M, 256);
    return (t * (t + 1) / 2) / (t * t);
}

size_t gemm_tc_splitk_bytes(const Gemm& g) {
    const bool pair = use_pairs(g);
    const int bm = pair ? 256 : BM, bn = pair ? P_BN : (g.N > 128 ? 256 : 128);
    const int tiles = ceil_div(g.M, bm) * ceil_div(g.N, bn);
    const int s = pick_splits(g, tiles, ceil_div(g.K, BK), pair ? num_sms() / 2 : num_sms());
    return s > 1 ? (size_t)s * g.batch * g.M * g.N * 4 : 0;
}

int gemm_tc(const Gemm& g, void* ws, size_t ws_bytes, cudaStream_t s) {
    if (!gemm_tc_supported(g)) return set_error(NC_ERR_UNSUPPORTED, "gemm_tc: unsupported operands");
    const bool pair = use_pairs(g);
    const int bm = pair ? 256 : BM;
    const int bn = pair ? P_BN : (g.N > 128 ? 256 : 128);
    TcParams p{};
    p.M = g.M; p.N = g.N; p.K = g.K; p.batch = g.batch;
    p.tiles_m = ceil_div(g.M, bm);
    p.tiles_n = ceil_div(g.N, bn);
    p.num_kb = ceil_div(g.K, BK);
    p.sym = g.sym && pair && g.M == g.N && g.epi == EPI_STORE && !g.a_t;
    p.splits = p.sym ? 1 : pick_splits(g, p.tiles_m * p.tiles_n, p.num_kb, pair ? num_sms() / 2 : num_sms());
    size_t need = p.splits > 1 ? (size_t)p.splits * g.batch * g.M * g.N * 4 : 0;
    if (need > ws_bytes || ws == nullptr) p.splits = 1;
    p.units = p.sym ? (long)p.tiles_m * (p.tiles_m + 1) / 2 * g.batch
                    : (long)p.tiles_m * p.tiles_n * p.splits * g.batch;
    p.C = g.C; p.ldc = g.ldc; p.sC = g.sC; p.c_dtype = g.c_dtype;
    p.aux = g.aux; p.ldaux = g.ldaux; p.sAux = g.sAux; p.aux_dtype = g.aux_dtype;
    p.alpha = g.alpha; p.beta = g.beta; p.epi = g.epi;
    p.ws = p.splits > 1 ? reinterpret_cast<float*>(ws) : nullptr;
    p.flag = g.flag;
    p.rope = g.rope; p.rope_T = g.rope_T; p.rope_cols = g.rope_cols; p.rope_ld = g.rope_ld; p.delta = g.delta;
    p.lse_part = g.lse_part;
    p.dot_out = g.dot_out;
    p.nb_r = g.nb_r; p.nb_part = g.nb_part; p.nb_nparts = g.nb_nparts; p.nb_inv_d = g.nb_inv_d;
    p.nb_gin = g.nb_gin; p.nb_gt = g.nb_gt;

    // the auxiliary matrix by TMA (32 x 32 blocks, 128 / 64-byte swizzle) when the
    // epilogue reads one and its layout allows the copy
    CUtensorMap ma, mb, mx;
    const bool reads_aux = (g.epi == EPI_STORE && g.aux && g.beta != 0.f) || g.epi == EPI_RELU2_BWD ||
                           g.epi == EPI_DELTA || g.epi == EPI_NORMB;
    const int xes = g.aux_dtype == NC_FP32 ? 4 : 2;
    if (reads_aux && p.splits == 1 && (g.ldaux * xes) % 16 == 0 && (g.batch <= 1 || (g.sAux * xes) % 16 == 0)) {
        NC_TRY(make_map_x(&mx, g.aux, g.aux_dtype, g.N, g.M, g.batch, g.ldaux, g.sAux));
        p.aux_tma = 1;
    }
    if (!g.a_t) NC_TRY(make_map(&ma, g.A, g.K, g.M, g.batch, g.lda, g.sA, 64, BM));
    else        NC_TRY(make_map(&ma, g.A, g.M, g.K, g.batch, g.lda, g.sA, 64, 64));
    if (!g.b_t) NC_TRY(make_map(&mb, g.B, g.K, g.N, g.batch, g.ldb, g.sB, 64, pair ? 128 : bn));
    else        NC_TRY(make_map(&mb, g.B, g.N, g.K, g.batch, g.ldb, g.sB, 64, 64));
    if (!p.aux_tma) mx = ma;   // unused

    int rc;
    if (pair) {
        const int ef = epi_family(g.epi, g.dot_out != nullptr);
        if (p.sym && !g.a_t) rc = g.b_t ? launch2<false, true, true>(ma, mb, mx, p, s)
                                        : launch2<false, false, true>(ma, mb, mx, p, s);
        else if (ef == EF_ROPE) rc = launch2<false, false, false, EF_ROPE>(ma, mb, mx, p, s);
        else if (ef == EF_LSE) rc = launch2<false, false, false, EF_LSE>(ma, mb, mx, p, s);
        else if (ef == EF_DELTA) rc = launch2<false, true, false, EF_DELTA>(ma, mb, mx, p, s);
        else if (ef == EF_NB) rc = launch2<false, true, false, EF_NB>(ma, mb, mx, p, s);
        else if (ef == EF_DOT) rc = launch2<false, true, false, EF_DOT>(ma, mb, mx, p, s);
        else if (!g.a_t && !g.b_t) rc = launch2<false, false>(ma, mb, mx, p, s);
        else if (!g.a_t && g.b_t) rc = launch2<false, true>(ma, mb, mx, p, s);
        else if (g.a_t && !g.b_t) rc = launch2<true, false>(ma, mb, mx, p, s);
        else rc = launch2<true, true>(ma, mb, mx, p, s);
    } else if (bn == 256) {
        if (!g.a_t && !g.b_t) rc = launch<256, false, false>(ma, mb, mx, p, s);
        else if (!g.a_t && g.b_t) rc = launch<256, false, true>(ma, mb, mx, p, s);
        else if (g.a_t && !g.b_t) rc = launch<256, true, false>(ma, mb, mx, p, s);
        else rc = launch<256, true, true>(ma, mb, mx, p, s);
    } else {
        if (!g.a_t && !g.b_t) rc = launch<128, false, false>(ma, mb, mx, p, s);
        else if (!g.a_t && g.b_t) rc = launch<128, false, true>(ma, mb, mx, p, s);
        else if (g.a_t && !g.b_t) rc = launch<128, true, false>(ma, mb, mx, p, s);
        else rc = launch<128, true, true>(ma, mb, mx, p, s);
    }
    NC_TRY(rc);
    if (p.splits > 1) {
        const long total = (long)g.batch * g.M * g.N;
        const bool vec = g.N % 4 == 0 && g.ldc % 4 == 0 && (!g.aux || g.ldaux % 4 == 0) &&
                         (g.batch <= 1 || (g.sC % 4 == 0 && (!g.aux || g.sAux % 4 == 0))) &&
                         (uintptr_t)g.C % 16 == 0 && (!g.aux || (uintptr_t)g.aux % 16 == 0) &&
                         total / 4 < (1L << 31) - 65536L * 256;
        if (vec) {
            const long quads = total / 4;
            const int blocks = (int)(quads / 256 < 8L * num_sms() ? ceil_div(quads, 256) : 8L * num_sms());
            splitk_reduce4_kernel<<<blocks, 256, 0, s>>>(p.ws, p.splits, g.batch * g.M, g.M, g.N, g.C, g.ldc,
                                                         g.sC, g.c_dtype, g.aux, g.ldaux, g.sAux, g.aux_dtype,
                                                         g.alpha, g.beta, g.epi);
        } else {
            splitk_reduce_kernel<<<ceil_div(total, 256), 256, 0, s>>>(
                p.ws, p.splits, g.batch, g.M, g.N, g.C, g.ldc, g.sC, g.c_dtype, g.aux, g.ldaux, g.sAux,
                g.aux_dtype, g.alpha, g.beta, g.epi);
        }
        note_launch();
        NC_LAUNCH_CHECK("splitk_reduce");
    }
    return NC_OK;
}

}  // namespace nc
