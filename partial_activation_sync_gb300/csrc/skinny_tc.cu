// Row-parallel forward + partial channel-reduce for few tokens (decode and small
// batches, up to a few hundred tokens) on the tensor cores, operands swapped.
//
// "Tensor-Parallelism with Partially Synchronized Activations" (Introduction,
// partial channel-reduce; inference with the partial reduce in place of the
// all-reduce).  With a few tokens the layer reads every weight once and the time
// is the weight stream, so the design goal is to keep HBM busy from every SM:
//
//   * one CTA per (128-channel block, shard r): it streams W_r[128 channels, k_t]
//     and the few token rows of X_r through a TMA ring and accumulates
//     D[channel, token] = W_r X_r^T in TMEM (tcgen05, M = 128 channels, N = 16..128
//     tokens: the token count is the MMA's narrow side);
//   * the t shard-CTAs of a channel block form one thread-block cluster: a channel
//     outside S is final in its own CTA (rank r's partial goes to Y[r]); for the
//     channels of S every CTA puts its fp32 partial tile in shared memory, and CTA
//     q sums a 1/t slice of the channels over the cluster (distributed shared
//     memory, rank order 0..t-1) and writes the sum to all t outputs;
//   * above 128 tokens the tokens are cut into chunks of 128, one cluster per
//     (channel block, chunk): the chunks of a block read the same weight tiles,
//     the first from HBM and the others mostly from L2.
//
// Warp roles: warp 0 issues the TMA loads, warp 1 owns TMEM and issues the MMAs,
// warps 2..5 read the accumulator back (warp w reads TMEM lanes 32*(w%4)..).
// Every wait is bounded (2 s of global time) and records CAAT_ERR_TIMEOUT.
#include <cuda.h>
#include <cuda_bf16.h>

#include <cstdlib>
#include <cstring>

#include "caat_internal.h"
#include "tc_ptx.cuh"

namespace caat {

__device__ int g_caat_skinny_error;

caat_status read_and_clear_skinny_error()
{
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_caat_skinny_error, sizeof(int)) != cudaSuccess) return CAAT_ERR_CUDA;
    if (v != 0) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_caat_skinny_error, &zero, sizeof(int)) != cudaSuccess) return CAAT_ERR_CUDA;
        return (caat_status)v;
    }
    return CAAT_OK;
}

namespace {

using namespace tc;

constexpr int CH = 128;                      // channels per CTA (MMA M)
constexpr int BK = 64;                       // k per stage (one 128-byte swizzled row)
constexpr int MAX_STAGES = 6;
// Ring depth by token tile: as deep as lets two CTAs share an SM (the 7B layers
// launch 256 CTAs on 152 SMs): 6 stages of 18 KB at NT = 16, 5 of 20 KB at 32,
// 4 of 24 KB at 64, 3 of 32 KB at 128.
template <int NT>
__host__ __device__ constexpr int stages() { return NT <= 16 ? 6 : (NT <= 32 ? 5 : (NT <= 64 ? 4 : 3)); }
constexpr int NUM_THREADS = 192;
constexpr int W_BYTES = CH * BK * 2;         // 16 KB
constexpr int MAX_T_SKINNY = 8;              // portable cluster size
constexpr int64_t SKINNY_MAX_N = 8192;       // token rows (chunks of 128 above 128 tokens)
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;

struct SkinnyCtl {
    uint64_t full[MAX_STAGES];
    uint64_t empty[MAX_STAGES];
    uint64_t acc_full;
    uint32_t tmem_base;
    int abort;
    uint32_t smask[CH / 32];                 // bit c: channel (block start + c) is in S
};

struct SkinnyParams {
    void *Y[MAX_T_SKINNY];
    int64_t ldy;
    int64_t N, h;
    int t, nkb;
    int vec;                                 // outputs take 16-byte stores (aligned rows)
    const int32_t *sel;
    int64_t n_sel;
    int prefetch_w;                          // weight tiles of the first stages before the wait
    int nchunks;                             // token chunks of NT rows (clusters per channel block)
};

template <int NT>
__host__ __device__ constexpr int x_bytes() { return NT * BK * 2; }

template <int NT>
constexpr size_t skinny_smem()
{
    return 1024 + (size_t)stages<NT>() * (W_BYTES + x_bytes<NT>()) + sizeof(SkinnyCtl);
}

__device__ __forceinline__ void fail(volatile int *abort)
{
    *abort = 1;
    atomicExch(&g_caat_skinny_error, (int)CAAT_ERR_TIMEOUT);
}

__device__ __forceinline__ float4 ld_cluster_v4(uint32_t addr)
{
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

__device__ __forceinline__ uint16_t to_bf16(float v)
{
    return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi)
{
    return (uint32_t)to_bf16(lo) | ((uint32_t)to_bf16(hi) << 16);
}

// 8 consecutive channels (ch0 .. ch0+7) of one output row: one 16-byte store
// when all 8 are wanted (mask bits set) and the row is aligned, else one 2-byte
// store per wanted channel below h.
__device__ __forceinline__ void store8(uint16_t *row, int64_t ch0, int64_t h, uint32_t want, bool vec,
                                       const float (&v)[8])
{
    if (vec && want == 0xffu && ch0 + 8 <= h) {
        uint4 w;
        w.x = pack2(v[0], v[1]);
        w.y = pack2(v[2], v[3]);
        w.z = pack2(v[4], v[5]);
        w.w = pack2(v[6], v[7]);
        *reinterpret_cast<uint4 *>(row + ch0) = w;
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (((want >> i) & 1u) && ch0 + i < h) row[ch0 + i] = to_bf16(v[i]);
    }
}

// grid: t CTAs per cluster (cluster rank = shard r) x one cluster per
// 128-channel block; NT = padded token count (MMA N), N <= NT.
template <int NT>
__global__ void __launch_bounds__(NUM_THREADS, 1)
rowpar_fwd_skinny_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                         const SkinnyParams p)
{
    constexpr int XB = x_bytes<NT>();
    constexpr int STAGES = stages<NT>();
    constexpr uint32_t TX = W_BYTES + XB;
    constexpr uint32_t TMEM_COLS = NT < 32 ? 32 : NT;
    constexpr uint32_t IDESC = idesc_bf16_f32(CH, NT);
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *smW = base;
    uint8_t *smX = base + STAGES * W_BYTES;
    SkinnyCtl *ctl = (SkinnyCtl *)(base + STAGES * (W_BYTES + XB));
    float *part = (float *)base;     // [NT][CH] fp32 partials, reusing the ring (W and X stages) after the last MMA
    volatile int *abort = &ctl->abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int t = p.t;
    const int r = t > 1 ? (int)cluster_ctarank() : 0;
    // cluster index -> (channel block, token chunk), the chunks of a channel block
    // adjacent so that they read its weight tiles at about the same time (from L2
    // after the first)
    const int ci = (int)(blockIdx.x / (unsigned)t);
    const int cb = ci / p.nchunks;
    const int64_t c0 = (int64_t)cb * CH;
    const int64_t tok0 = (int64_t)(ci % p.nchunks) * NT;
    const int ntok = p.N - tok0 < NT ? (int)(p.N - tok0) : NT;   // token rows of this chunk (>= 1)

    if (tid < CH / 32) ctl->smask[tid] = 0u;
    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&ctl->full[s]), 1);
            mbar_init(smem_u32(&ctl->empty[s]), 1);
        }
        mbar_init(smem_u32(&ctl->acc_full), 1);
        ctl->abort = 0;
        fence_mbar_init();
        prefetch_tmap(&tmX);
        prefetch_tmap(&tmW);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&ctl->tmem_base), TMEM_COLS);
        tmem_relinquish();
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = ctl->tmem_base;
    // Launched as a programmatic dependent, this grid may have started while the
    // previous one in the stream was still running: nothing above touched global
    // memory (the tensor maps are launch parameters).  Wait for it before the
    // first load or store, then let the next grid start its own setup.  With
    // prefetch_w the producer thread waits later, after it has issued the weight
    // tiles of the first ring stages (the caller guarantees that the previous
    // launch does not write the weights); the rest of warp 0 touches no memory.
    if (!(p.prefetch_w != 0 && warp == 0)) griddep_wait();
    griddep_launch_dependents();

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t ph = 0;
            int kb0 = 0;
            if (p.prefetch_w != 0) {
                // the first pass over the ring needs no empty-slot wait: weight
                // tiles now, then (after the previous grid) the token tiles
                const int pre = p.nkb < STAGES ? p.nkb : STAGES;
                for (int kb = 0; kb < pre; ++kb) {
                    const uint32_t fb = smem_u32(&ctl->full[kb]);
                    mbar_arrive_expect_tx(fb, TX);
                    tma_load_3d(smem_u32(smW + kb * W_BYTES), &tmW, fb, kb * BK, r, (int)c0);
                }
                griddep_wait();
                for (int kb = 0; kb < pre; ++kb)
                    tma_load_3d(smem_u32(smX + kb * XB), &tmX, smem_u32(&ctl->full[kb]), kb * BK, r, (int)tok0);
                kb0 = pre;
                stage = pre % STAGES;
                ph = pre == STAGES ? 1u : 0u;
            }
            for (int kb = kb0; kb < p.nkb; ++kb) {
                if (!mbar_wait(smem_u32(&ctl->empty[stage]), ph ^ 1u, abort, WAIT_LIMIT_NS)) {
                    fail(abort);
                    break;
                }
                const uint32_t fb = smem_u32(&ctl->full[stage]);
                mbar_arrive_expect_tx(fb, TX);
                tma_load_3d(smem_u32(smW + stage * W_BYTES), &tmW, fb, kb * BK, r, (int)c0);
                tma_load_3d(smem_u32(smX + stage * XB), &tmX, fb, kb * BK, r, (int)tok0);
                if (++stage == STAGES) { stage = 0; ph ^= 1u; }
            }
        }
    } else if (warp == 1) {
        // -------------------------------------------------------- MMA issuer
        if (lane == 0) {
            int stage = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int kb = 0; kb < p.nkb; ++kb) {
                if (!mbar_wait(smem_u32(&ctl->full[stage]), ph, abort, WAIT_LIMIT_NS)) {
                    fail(abort);
                    ok = false;
                    break;
                }
                fence_after_sync();
                const uint32_t a0 = smem_u32(smW + stage * W_BYTES);
                const uint32_t b0 = smem_u32(smX + stage * XB);
#pragma unroll
                for (int k = 0; k < BK / 16; ++k)
                    mma_f16(tmem, desc_kmajor_sw128(a0 + 32u * k), desc_kmajor_sw128(b0 + 32u * k), IDESC,
                            (kb == 0 && k == 0) ? 0u : 1u);
                mma_commit(smem_u32(&ctl->empty[stage]));
                if (++stage == STAGES) { stage = 0; ph ^= 1u; }
            }
            if (ok) mma_commit(smem_u32(&ctl->acc_full));
        }
    } else {
        // ---------------------------------------------------------- epilogue
        // Membership of this block's channels in S, built while the weights
        // stream in: every index of S is read once, eight independent loads per
        // thread in flight.
        const int e = tid - 64;
        if (p.sel == nullptr) {      // S = {0, ..., n_sel-1}
            if (e < CH / 32) {
                const int64_t lo = c0 + 32 * e;
                ctl->smask[e] = p.n_sel >= lo + 32 ? 0xffffffffu
                              : (p.n_sel <= lo ? 0u : ((1u << (uint32_t)(p.n_sel - lo)) - 1u));
            }
        } else {
            for (int64_t i0 = e; i0 < p.n_sel; i0 += 128 * 8) {
                int32_t v[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) v[u] = i0 + 128 * u < p.n_sel ? __ldg(p.sel + i0 + 128 * u) : -1;
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int64_t c = v[u];
                    if (c >= c0 && c < c0 + CH && c < p.h)
                        atomicOr(&ctl->smask[(c - c0) >> 5], 1u << ((c - c0) & 31));
                }
            }
        }
        asm volatile("bar.sync 1, 128;" ::: "memory");          // the four epilogue warps
        const bool any_s_e = t > 1 && (ctl->smask[0] | ctl->smask[1] | ctl->smask[2] | ctl->smask[3]) != 0u;
        const int q = warp & 3;                                  // TMEM lane quarter
        const int cl = 32 * q + lane;                            // channel within the block
        bool ok = mbar_wait(smem_u32(&ctl->acc_full), 0u, abort, WAIT_LIMIT_NS);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) fail(abort);
        if (ok) {
            // accumulator -> part[token][channel] (fp32; lane = channel, so the
            // 32 lanes of a warp write one 128-byte row segment)
            fence_after_sync();
#pragma unroll
            for (int half = 0; half < (NT + 31) / 32; ++half) {
                uint32_t v[32];
                tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + 32u * half, v);
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (32 * half + j < NT) part[(32 * half + j) * CH + cl] = __uint_as_float(v[j]);
            }
        }
        asm volatile("bar.sync 1, 128;" ::: "memory");
        if (ok) {
            // this rank's channels outside S, row by row, 8 channels per store
            uint16_t *yr = nullptr;
#pragma unroll
            for (int qq = 0; qq < MAX_T_SKINNY; ++qq)
                if (qq == r) yr = (uint16_t *)p.Y[qq];
            for (int it = e; it < ntok * (CH / 8); it += 128) {
                const int tok = it / (CH / 8), cl0 = 8 * (it % (CH / 8));
                const int64_t ch0 = c0 + cl0;
                if (ch0 >= p.h) continue;
                const uint32_t sbits = any_s_e ? (ctl->smask[cl0 >> 5] >> (cl0 & 31)) & 0xffu : 0u;
                if (sbits == 0xffu) continue;
                const float4 a = *reinterpret_cast<const float4 *>(part + tok * CH + cl0);
                const float4 b = *reinterpret_cast<const float4 *>(part + tok * CH + cl0 + 4);
                const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
                store8(yr + (tok0 + tok) * p.ldy, ch0, p.h, ~sbits & 0xffu, p.vec != 0, v);
            }
        }
    }

    // ---- the S channels: sum the t partial tiles over the cluster
    __syncthreads();                 // the mask is complete for every warp
    const bool any_s = t > 1 && (ctl->smask[0] | ctl->smask[1] | ctl->smask[2] | ctl->smask[3]) != 0u;
    if (any_s) {
        cluster_sync();              // every CTA's partial tile is in its shared memory
        if (warp >= 2 && !*abort) {
            // CTA r sums channels [lo, hi) of the block: all t partials of 8
            // channels are loaded before they are added in rank order 0..t-1
            const int e = tid - 64;
            const int lo = (r * CH) / t, hi = ((r + 1) * CH) / t;
            const uint32_t my_part = smem_u32(part);
            const int g0 = lo / 8, g1 = (hi + 7) / 8;        // 8-channel groups touching [lo, hi)
            const int ng = g1 - g0;
            for (int it = e; it < ntok * ng; it += 128) {
                const int tok = it / ng, cl0 = 8 * (g0 + it % ng);
                const int64_t ch0 = c0 + cl0;
                if (ch0 >= p.h) continue;
                // this CTA's share of the group: channels in [lo, hi) and in S
                uint32_t own = 0u;
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (cl0 + i >= lo && cl0 + i < hi) own |= 1u << i;
                const uint32_t want = own & ((ctl->smask[cl0 >> 5] >> (cl0 & 31)) & 0xffu);
                if (want == 0u) continue;
                const uint32_t off = my_part + (uint32_t)(tok * CH + cl0) * 4u;
                float4 va[MAX_T_SKINNY], vb[MAX_T_SKINNY];
#pragma unroll
                for (int qq = 0; qq < MAX_T_SKINNY; ++qq) {
                    if (qq < t) {
                        va[qq] = ld_cluster_v4(map_to_cta(off, (uint32_t)qq));
                        vb[qq] = ld_cluster_v4(map_to_cta(off + 16u, (uint32_t)qq));
                    }
                }
                float v[8] = {va[0].x, va[0].y, va[0].z, va[0].w, vb[0].x, vb[0].y, vb[0].z, vb[0].w};
#pragma unroll
                for (int qq = 1; qq < MAX_T_SKINNY; ++qq) {
                    if (qq < t) {
                        v[0] = v[0] + va[qq].x; v[1] = v[1] + va[qq].y;
                        v[2] = v[2] + va[qq].z; v[3] = v[3] + va[qq].w;
                        v[4] = v[4] + vb[qq].x; v[5] = v[5] + vb[qq].y;
                        v[6] = v[6] + vb[qq].z; v[7] = v[7] + vb[qq].w;
                    }
                }
#pragma unroll
                for (int qq = 0; qq < MAX_T_SKINNY; ++qq)
                    if (qq < t) store8((uint16_t *)p.Y[qq] + (tok0 + tok) * p.ldy, ch0, p.h, want, p.vec != 0, v);
            }
        }
        cluster_sync();              // no CTA leaves while another reads its tile
    }

    fence_before_sync();
    __syncthreads();
    if (*abort) {
        // let copies and MMAs already in flight land before TMEM and shared
        // memory go away
        if (tid == 0) {
            const uint64_t t0 = globaltimer();
            while (globaltimer() - t0 < 2000000ull) { }
        }
        __syncthreads();
    }
    if (warp == 1) {
        __syncwarp();
        fence_after_sync();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

template <int NT>
caat_status launch_nt(const CUtensorMap &tmX, const CUtensorMap &tmW, const SkinnyParams &p, int num_cb,
                      cudaStream_t s)
{
    auto kern = rowpar_fwd_skinny_kernel<NT>;
    constexpr size_t smem = skinny_smem<NT>();
    static_assert(2 * (smem + 1024) <= 228 * 1024, "two CTAs per SM (1 KB reserved each)");
    static_assert((size_t)NT * CH * 4 <= (size_t)stages<NT>() * (W_BYTES + x_bytes<NT>()), "partials fit in the ring");
    if (prepare_kernel_smem((const void *)kern, (int)smem) != CAAT_OK) return CAAT_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)p.t;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3((unsigned)(p.t * num_cb * p.nchunks));
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (max_active_clusters((const void *)kern, cfg) < 1) return CAAT_ERR_UNSUPPORTED;
    // A programmatic dependent of the previous launch in the stream (CAAT_PDL=0:
    // a plain launch): its CTAs may be set up while that grid finishes; the
    // kernel waits for it before touching memory.
    const char *pdl_env = std::getenv("CAAT_PDL");
    if (pdl_env == nullptr || std::strcmp(pdl_env, "0") != 0) {
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.numAttrs = 2;
    }
    if (cudaLaunchKernelEx(&cfg, kern, tmX, tmW, p) != cudaSuccess) return CAAT_ERR_CUDA;
    note_launch("rowpar_fwd_skinny_tc");
    return cudaGetLastError() == cudaSuccess ? CAAT_OK : CAAT_ERR_CUDA;
}

}  // namespace

caat_status launch_rowpar_fwd_skinny(int t, int64_t N, int64_t K, int64_t h, const void *X, int64_t ldx,
                                     const void *W, int64_t ldw, const MutPtrs &Y, int64_t ldy,
                                     const int32_t *sel, int64_t n_sel, cudaStream_t s)
{
    const int64_t kt = K / t;
    if (t < 1 || t > MAX_T_SKINNY || N < 1 || N > SKINNY_MAX_N || kt < BK || kt % 8 != 0) return CAAT_ERR_UNSUPPORTED;
    if (ldx % 8 != 0 || ldw % 8 != 0 || h < 1 || h > (int64_t)INT32_MAX / 2) return CAAT_ERR_UNSUPPORTED;
    if ((uintptr_t)X % 16 != 0 || (uintptr_t)W % 16 != 0) return CAAT_ERR_UNSUPPORTED;
    if (kt > (int64_t)INT32_MAX / 2 || N * ldy > (int64_t)INT32_MAX) return CAAT_ERR_UNSUPPORTED;
    const int nt = N <= 16 ? 16 : (N <= 32 ? 32 : (N <= 64 ? 64 : 128));
    CUtensorMap tmX, tmW;
    {
        const uint64_t dims[3] = {(uint64_t)kt, (uint64_t)t, (uint64_t)N};
        const uint64_t str[2] = {(uint64_t)kt * 2, (uint64_t)ldx * 2};
        const uint32_t box[3] = {BK, 1, (uint32_t)nt};
        if (!encode_tmap(&tmX, X, 3, dims, str, box)) return CAAT_ERR_UNSUPPORTED;
    }
    {
        const uint64_t dims[3] = {(uint64_t)kt, (uint64_t)t, (uint64_t)h};
        const uint64_t str[2] = {(uint64_t)kt * 2, (uint64_t)ldw * 2};
        const uint32_t box[3] = {BK, 1, CH};
        if (!encode_tmap(&tmW, W, 3, dims, str, box)) return CAAT_ERR_UNSUPPORTED;
    }
    SkinnyParams p{};
    bool vec = ldy % 8 == 0;
    for (int q = 0; q < t; ++q) {
        p.Y[q] = Y.p[q];
        vec = vec && (uintptr_t)Y.p[q] % 16 == 0;
    }
    p.vec = vec ? 1 : 0;
    p.ldy = ldy;
    p.N = N;
    p.h = h;
    p.t = t;
    p.nkb = (int)((kt + BK - 1) / BK);
    p.sel = sel;
    p.n_sel = n_sel;
    const char *pw_env = std::getenv("CAAT_PDL_WEIGHTS");
    p.prefetch_w = pw_env != nullptr && std::strcmp(pw_env, "1") == 0;
    p.nchunks = (int)((N + nt - 1) / nt);
    const int64_t num_cb = (h + CH - 1) / CH;
    if (num_cb * t * p.nchunks > INT32_MAX) return CAAT_ERR_UNSUPPORTED;
    // Token chunks re-read each weight tile from L2, and more than two CTAs per SM
    // run in several waves: at the 7B shapes (256 CTAs a chunk) two chunks are
    // faster than the tile kernel, three are slower.
    if (p.nchunks > 1 && num_cb * t * p.nchunks > 4 * (int64_t)num_sms()) return CAAT_ERR_UNSUPPORTED;
    switch (nt) {
    case 16: return launch_nt<16>(tmX, tmW, p, (int)num_cb, s);
    case 32: return launch_nt<32>(tmX, tmW, p, (int)num_cb, s);
    case 64: return launch_nt<64>(tmX, tmW, p, (int)num_cb, s);
    default: return launch_nt<128>(tmX, tmW, p, (int)num_cb, s);
    }
}

}  // namespace caat
