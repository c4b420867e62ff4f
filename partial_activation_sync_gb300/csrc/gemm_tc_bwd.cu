// Backward GEMMs of the fused row-parallel layer on the 5th-generation tensor
// core (sm_103a): one grouped, persistent tcgen05 GEMM per gradient.
//
// "Tensor-Parallelism with Partially Synchronized Activations", Introduction:
// forward and backward must agree.  With dY_r the (partially reduced) gradient
// of rank r's output, the rank's shard of the input gradient and of the weight
// gradient are
//   dX[:, shard r]      = dY_r W_r^T   (M = tokens,   N = k_t, K = h)
//   dW[shard r, :]^T    = dY_r^T X_r   (M = channels, N = k_t, K = tokens)
// Both are batched over the t ranks.  The operand that carries the rank's K
// shard (W_r or X_r) is read through one 3-D tensor map (k within shard, shard,
// row); dY_r through one 2-D tensor map per rank.  W_r^T and X_r are MN-major
// operands (their n index is contiguous in memory), dY_r^T too, so the MMA reads
// them with the MN-major shared-memory layout instead of transposing in memory.
//
// Same machinery as the forward kernel: TMA into a ring of stages (warp 0), one
// thread issuing tcgen05.mma into two alternating TMEM accumulators (warp 1),
// four epilogue warps converting to bf16 and storing.  Above one 128-row block
// the tiles are 256 rows on a CTA pair (cta_group::2), which halves the operand
// bytes each SM pulls per FLOP of B.  Every wait is bounded.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <cstdlib>
#include <cstring>

#include "caat_internal.h"
#include "tc_ptx.cuh"

namespace caat {

// This file's own device error word (device symbols are not shared across
// translation units in this build); read through read_and_clear_bwd_error().
__device__ int g_bwd_dev_error;

caat_status read_and_clear_bwd_error()
{
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_bwd_dev_error, sizeof(int)) != cudaSuccess) return CAAT_ERR_CUDA;
    if (v != 0) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_bwd_dev_error, &zero, sizeof(int)) != cudaSuccess) return CAAT_ERR_CUDA;
        return (caat_status)v;
    }
    return CAAT_OK;
}

namespace {

using namespace tc;

constexpr int BM = 128, BK = 64, MAX_BN = 256;
constexpr int MAX_STAGES = 6;
constexpr int A_BYTES = BM * BK * 2;
constexpr int NUM_THREADS = 192;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;
constexpr int MAX_T_TC = 16;
constexpr int STG_BYTES = 32 * 128;          // 32 rows x 64 bf16 columns

struct TmapArray {
    CUtensorMap m[MAX_T_TC];
};

struct SmemCtl {
    uint64_t full[MAX_STAGES];
    uint64_t empty[MAX_STAGES];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint32_t tmem_base;
    int abort;
};

// The ring: stages of A (128 x 64) + B (BN x 64); 4 stages of the widest tiles
// fit.  Narrower tiles take more stages (BN = 192: 5 stages and one staging
// buffer per epilogue warp; BN <= 128: 6 stages and two), which keeps more
// operand bytes in flight -- these short-K GEMMs otherwise wait on their ring.
constexpr size_t SMEM_LIMIT = 227 * 1024;
struct Ring {
    int stages, stage_bytes, nbuf;
};
inline Ring ring_for(int BN, bool deep)
{
    Ring g;
    g.stage_bytes = A_BYTES + BN * BK * 2;
    g.stages = !deep ? 4 : (BN <= 128 ? 6 : (BN <= 192 ? 5 : 4));
    g.nbuf = (deep && BN > 128 && BN <= 192) ? 1 : 2;
    return g;
}
// CTA pairs: A (128 x 64) + this CTA's half of B (at most 128 x 64) per stage
inline Ring ring_for_pair()
{
    Ring g;
    g.stage_bytes = A_BYTES + (MAX_BN / 2) * BK * 2;
    g.stages = 6;
    g.nbuf = 2;
    return g;
}
inline size_t ring_smem(const Ring &g)
{
    return 1024 + (size_t)g.stages * g.stage_bytes + 4 * g.nbuf * STG_BYTES + sizeof(SmemCtl);
}

struct GemmParams {
    int64_t M, Nn, Kk;  // per-rank GEMM
    int t, num_m, num_n, nkb, units;
    int BN;             // column tile width
    int s_blocks;       // 64-channel blocks of the gradient read from the reduced sum (smap)
    int ksplit, kbps;   // K range split in ksplit parts of kbps k-blocks (RED only)
    int stages, stage_bytes, nbuf;   // the ring (see ring_for)
    uint32_t idesc;
};

__device__ __forceinline__ void fail(volatile int *abort)
{
    *abort = 1;
    atomicExch(&g_bwd_dev_error, (int)CAAT_ERR_TIMEOUT);
}

__device__ __forceinline__ uint32_t pack_bf16x2(uint32_t lo_f32, uint32_t hi_f32)
{
    const __nv_bfloat162 v = __floats2bfloat162_rn(__uint_as_float(lo_f32), __uint_as_float(hi_f32));
    return *reinterpret_cast<const uint32_t *>(&v);
}

// One work unit: rank r, 128-row block mb of this CTA, column tile nb,
// k-blocks [kb_lo, kb_hi).  With CTA pairs a unit is a 256-row block whose
// halves are the two CTAs' row blocks.  Units run the K parts of every column
// tile of a row block, then the next row block, then the next rank: the units
// dealt to neighbouring workers share their A rows.
struct Unit {
    int r, mb, nb, kb_lo, kb_hi;
};

template <bool PAIR>
__device__ __forceinline__ Unit decode_unit(int u, const GemmParams &p, uint32_t crank)
{
    Unit x;
    const int num_mu = PAIR ? (p.num_m + 1) / 2 : p.num_m;
    const int ks = u % p.ksplit;
    int v = u / p.ksplit;
    x.nb = v % p.num_n;
    v /= p.num_n;
    const int mu = v % num_mu;
    x.r = v / num_mu;
    x.mb = PAIR ? 2 * mu + (int)crank : mu;
    x.kb_lo = ks * p.kbps;
    x.kb_hi = min(p.nkb, x.kb_lo + p.kbps);
    return x;
}

// A_MN: A is MN-major (dW: dY_r^T); otherwise K-major (dX: dY_r).  B is MN-major.
// RED: the K range is split over several CTAs and each adds its fp32 partial
// into an fp32 array with a TMA reduce-add (cmap is then an fp32 map);
// otherwise the tile is rounded to bf16 and stored.
// PAIR: a CTA pair (cta_group::2) computes a 256-row tile.  Each CTA loads its
// own 128 rows of A and its half of the tile's columns of B; both halves land
// on the even CTA's barriers, whose single thread issues the MMAs for the pair.
// Each CTA's TMEM then holds its 128 rows of the accumulator, which its own
// epilogue warps store.  Per SM this halves the B bytes per FLOP.  Pairs take
// 256-column tiles only: each half is two whole 64-column boxes.
template <bool A_MN, bool RED, bool PAIR>
__global__ void __launch_bounds__(NUM_THREADS, 1)
grouped_gemm_tc_kernel(const __grid_constant__ TmapArray amaps, const __grid_constant__ CUtensorMap smap,
                       const __grid_constant__ CUtensorMap bmap, const __grid_constant__ CUtensorMap cmap,
                       const GemmParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *staging = base + p.stages * p.stage_bytes;
    SmemCtl *ctl = (SmemCtl *)(staging + 4 * p.nbuf * STG_BYTES);
    volatile int *abort = &ctl->abort;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t crank = PAIR ? cluster_ctarank() : 0u;
    const bool is_leader = crank == 0u;

    if (tid == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(smem_u32(&ctl->full[s]), 1);
            mbar_init(smem_u32(&ctl->empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&ctl->acc_full[b]), 1);
            mbar_init(smem_u32(&ctl->acc_empty[b]), PAIR ? 256 : 128);
        }
        ctl->abort = 0;
        fence_mbar_init();
        prefetch_tmap(&bmap);
    }
    if (PAIR) cluster_sync();        // the peer's barriers exist before anything signals them
    if (warp == 1) {
        if (PAIR) {
            tmem_alloc_pair(smem_u32(&ctl->tmem_base), TMEM_COLS);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(smem_u32(&ctl->tmem_base), TMEM_COLS);
            tmem_relinquish();
        }
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = ctl->tmem_base;
    // a programmatic dependent of the previous launch in the stream: wait for it
    // before the first global read or write, then let the next grid set up
    griddep_wait();
    griddep_launch_dependents();
    // units are dealt round-robin to the workers (CTAs, or CTA pairs)
    const int worker = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
    const int nworkers = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;

    if (warp == 0) {
        if (lane == 0) {
            int stage = 0;
            uint32_t ph = 0;
            for (int u = worker; u < p.units; u += nworkers) {
                const Unit x = decode_unit<PAIR>(u, p, crank);
                const int m0 = x.mb * BM;
                // B columns this CTA loads: all BN, or its half of them
                const int half = PAIR ? p.BN / 2 : p.BN;
                const int nc0 = x.nb * p.BN + (int)crank * half;
                const uint32_t bytes = (uint32_t)(A_BYTES + half * BK * 2);
                for (int kb = x.kb_lo; kb < x.kb_hi; ++kb) {
                    if (!mbar_wait(smem_u32(&ctl->empty[stage]), ph ^ 1u, abort, WAIT_LIMIT_NS)) {
                        fail(abort);
                        goto done;
                    }
                    const uint32_t fb = smem_u32(&ctl->full[stage]);
                    uint32_t fbar = fb;
                    if (PAIR) {
                        fbar = map_to_cta(fb, 0);
                        if (is_leader) mbar_arrive_expect_tx(fb, 2u * bytes);
                    } else {
                        mbar_arrive_expect_tx(fb, bytes);
                    }
                    uint8_t *sa = base + stage * p.stage_bytes;
                    uint8_t *sb = sa + A_BYTES;
                    const int k0 = kb * BK;
                    // gradient channels below s_blocks*64 come from the reduced sum
                    // (shared by all ranks), the rest from rank r's own gradient,
                    // whose map starts at channel s_blocks*64
                    const int sc = p.s_blocks * 64;
                    if (A_MN) {
#pragma unroll
                        for (int i = 0; i < 2; ++i) {
                            const int c = m0 + 64 * i;
                            const CUtensorMap *am = c < sc ? &smap : &amaps.m[x.r];
                            const int cc = c < sc ? c : c - sc;
                            if (PAIR) tma_load_2d_pair(smem_u32(sa + 8192 * i), am, fbar, cc, k0);
                            else tma_load_2d(smem_u32(sa + 8192 * i), am, fbar, cc, k0);
                        }
                    } else {
                        const CUtensorMap *am = k0 < sc ? &smap : &amaps.m[x.r];
                        const int kk = k0 < sc ? k0 : k0 - sc;
                        if (PAIR) tma_load_2d_pair(smem_u32(sa), am, fbar, kk, m0);
                        else tma_load_2d(smem_u32(sa), am, fbar, kk, m0);
                    }
                    for (int i = 0; i < half / 64; ++i) {      // 64 columns x 64 rows each
                        if (PAIR) tma_load_3d_pair(smem_u32(sb + i * 8192), &bmap, fbar, nc0 + 64 * i, x.r, k0);
                        else tma_load_3d(smem_u32(sb + i * 8192), &bmap, fbar, nc0 + 64 * i, x.r, k0);
                    }
                    if (++stage == p.stages) { stage = 0; ph ^= 1u; }
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && is_leader) {
            int stage = 0;
            uint32_t ph = 0, au = 0;
            for (int u = worker; u < p.units; u += nworkers) {
                const Unit x = decode_unit<PAIR>(u, p, crank);
                const uint32_t b = au & 1u;
                if (!mbar_wait(smem_u32(&ctl->acc_empty[b]), ((au >> 1) & 1u) ^ 1u, abort, WAIT_LIMIT_NS)) {
                    fail(abort);
                    goto done;
                }
                fence_after_sync();
                const uint32_t d = tmem + b * (uint32_t)p.BN;
                for (int kb = x.kb_lo; kb < x.kb_hi; ++kb) {
                    if (!mbar_wait(smem_u32(&ctl->full[stage]), ph, abort, WAIT_LIMIT_NS)) {
                        fail(abort);
                        goto done;
                    }
                    fence_after_sync();
                    const uint32_t a0 = smem_u32(base + stage * p.stage_bytes);
                    const uint32_t b0 = a0 + A_BYTES;
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k) {
                        const uint64_t ad = A_MN ? desc_sw128(a0 + 2048u * k, 8192u, 1024u)
                                                 : desc_kmajor_sw128(a0 + 32u * k);
                        const uint64_t bd = desc_sw128(b0 + 2048u * k, 8192u, 1024u);
                        const uint32_t acc = (kb == x.kb_lo && k == 0) ? 0u : 1u;
                        if (PAIR) mma_f16_pair(d, ad, bd, p.idesc, acc);
                        else mma_f16(d, ad, bd, p.idesc, acc);
                    }
                    if (PAIR) mma_commit_pair_mc(smem_u32(&ctl->empty[stage]), (uint16_t)3u);
                    else mma_commit(smem_u32(&ctl->empty[stage]));
                    if (++stage == p.stages) { stage = 0; ph ^= 1u; }
                }
                if (PAIR) mma_commit_pair_mc(smem_u32(&ctl->acc_full[b]), (uint16_t)3u);
                else mma_commit(smem_u32(&ctl->acc_full[b]));
                ++au;
            }
        }
    } else {
        const int q = warp & 3;
        const uint32_t lane_off = (uint32_t)(32 * q) << 16;
        uint32_t au = 0;
        int sbuf = 0;
        for (int u = worker; u < p.units; u += nworkers) {
            const Unit x = decode_unit<PAIR>(u, p, crank);
            const int64_t n0 = (int64_t)x.nb * p.BN;
            const uint32_t b = au & 1u;
            bool ok = mbar_wait(smem_u32(&ctl->acc_full[b]), (au >> 1) & 1u, abort, WAIT_LIMIT_NS);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) {
                fail(abort);
                goto done;
            }
            fence_after_sync();
            const uint32_t tb = tmem + lane_off + b * (uint32_t)p.BN;
            // 32 rows x 64 columns per bulk store; the output map (column within
            // shard, shard, row) clips columns past k_t and rows past M
            const int y = x.mb * BM + 32 * q;
            if (RED) {
                // fp32 partial: 32 rows x 32 columns (128-byte rows) per reduce-add;
                // 64 columns are read from TMEM under one wait (BN is a multiple of 64)
#pragma unroll 1
                for (int c64 = 0; c64 < p.BN / 64; ++c64) {
                    if (n0 + 64 * c64 >= p.Nn) break;
                    uint32_t vv[2][32];
                    tmem_ld32x2(tb + 64u * c64, tb + 64u * c64 + 32u, vv[0], vv[1]);
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        const int64_t c0 = n0 + 64 * c64 + 32 * hf;
                        if (c0 >= p.Nn) break;         // same for the whole warp
                        uint8_t *stg = staging + (q * p.nbuf + sbuf) * STG_BYTES;
                        const uint32_t stg_a = smem_u32(stg);
                        if (++sbuf == p.nbuf) sbuf = 0;
                        if (lane == 0) {
                            if (p.nbuf > 1) bulk_wait_read1(); else bulk_wait_read0();
                        }
                        __syncwarp();
                        uint4 *rowp = reinterpret_cast<uint4 *>(stg + lane * 128);
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            rowp[j ^ (lane & 7)] =
                                make_uint4(vv[hf][4 * j], vv[hf][4 * j + 1], vv[hf][4 * j + 2], vv[hf][4 * j + 3]);
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0 && y < p.M) {
                            tma_reduce_add_3d(&cmap, stg_a, (int)c0, x.r, y);
                            bulk_commit();
                        }
                    }
                }
            }
#pragma unroll 1
            for (int c64 = 0; c64 < p.BN / 64 && !RED; ++c64) {
                const int64_t c0 = n0 + 64 * c64;
                if (c0 >= p.Nn) break;
                uint32_t v0[32], v1[32];
                tmem_ld32x2(tb + 64u * c64, tb + 64u * c64 + 32u, v0, v1);
                uint32_t w[32];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    w[i] = pack_bf16x2(v0[2 * i], v0[2 * i + 1]);
                    w[16 + i] = pack_bf16x2(v1[2 * i], v1[2 * i + 1]);
                }
                uint8_t *stg = staging + (q * p.nbuf + sbuf) * STG_BYTES;
                const uint32_t stg_a = smem_u32(stg);
                if (++sbuf == p.nbuf) sbuf = 0;
                if (lane == 0) {                    // the store that last used this buffer has read it
                    if (p.nbuf > 1) bulk_wait_read1(); else bulk_wait_read0();
                }
                __syncwarp();
                uint4 *rowp = reinterpret_cast<uint4 *>(stg + lane * 128);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    rowp[j ^ (lane & 7)] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0 && y < p.M) {
                    tma_store_3d(&cmap, stg_a, (int)c0, x.r, y);
                    bulk_commit();
                }
            }
            fence_before_sync();
            // release the accumulator to the MMA issuer (the even CTA's barrier)
            const uint32_t eb = smem_u32(&ctl->acc_empty[b]);
            if (PAIR) mbar_arrive_cluster(map_to_cta(eb, 0));
            else mbar_arrive(eb);
            ++au;
        }
    }

done:
    if (warp >= 2 && lane == 0) bulk_wait0();
    fence_before_sync();
    __syncthreads();
    if (*abort) {
        if (tid == 0) {
            const uint64_t t0 = globaltimer();
            while (globaltimer() - t0 < 2000000ull) { }
        }
        __syncthreads();
    }
    if (PAIR) cluster_sync();        // neither CTA leaves while its peer may still signal it
    if (warp == 1) {
        __syncwarp();
        fence_after_sync();
        if (PAIR) tmem_dealloc_pair(tmem, TMEM_COLS);
        else tmem_dealloc(tmem, TMEM_COLS);
    }
}

// smallest multiple of 64 (<= 256) that covers n in as few tiles as possible
int pick_bn(int64_t n)
{
    const int64_t tiles = (n + MAX_BN - 1) / MAX_BN;
    const int64_t per = (n + tiles - 1) / tiles;
    return (int)((per + 63) / 64 * 64);
}

template <bool A_MN, bool RED, bool PAIR>
caat_status launch_grouped(const TmapArray &amaps, const CUtensorMap &smap, const CUtensorMap &bmap,
                           const CUtensorMap &cmap, GemmParams &p, cudaStream_t s, const char *name)
{
    if (p.units <= 0) return CAAT_OK;
    auto kern = grouped_gemm_tc_kernel<A_MN, RED, PAIR>;
    // the ring for this tile width (CAAT_BWD_RING=4 keeps 4 stages at every width)
    const char *ring_env = std::getenv("CAAT_BWD_RING");
    const Ring g = PAIR ? ring_for_pair() : ring_for(p.BN, !(ring_env != nullptr && ring_env[0] == '4'));
    p.stages = g.stages;
    p.stage_bytes = g.stage_bytes;
    p.nbuf = g.nbuf;
    const size_t smem = ring_smem(g);
    if (smem > SMEM_LIMIT || p.stages > MAX_STAGES) return CAAT_ERR_UNSUPPORTED;
    if (prepare_kernel_smem((const void *)kern, (int)SMEM_LIMIT) != CAAT_OK) return CAAT_ERR_CUDA;
    // a programmatic dependent of the previous launch in the stream (CAAT_PDL=0: a
    // plain launch); the kernel waits for that grid before touching memory
    const char *pdl_env = std::getenv("CAAT_PDL");
    const bool pdl = pdl_env == nullptr || std::strcmp(pdl_env, "0") != 0;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 0;
    if (PAIR) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.numAttrs = 1;
        int pairs = num_sms() / 2;
        cfg.gridDim = dim3(2 * pairs);
        const int active = max_active_clusters((const void *)kern, cfg);
        if (active < 1) return CAAT_ERR_UNSUPPORTED;
        if (active < pairs) pairs = active;
        if (pairs > p.units) pairs = p.units;
        cfg.gridDim = dim3(2 * pairs);
    } else {
        cfg.gridDim = dim3(p.units < num_sms() ? p.units : num_sms());
    }
    if (pdl) {
        attr[cfg.numAttrs].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[cfg.numAttrs].val.programmaticStreamSerializationAllowed = 1;
        ++cfg.numAttrs;
    }
    if (cudaLaunchKernelEx(&cfg, kern, amaps, smap, bmap, cmap, p) != cudaSuccess) return CAAT_ERR_CUDA;
    note_launch(name);
    return cudaGetLastError() == cudaSuccess ? CAAT_OK : CAAT_ERR_CUDA;
}

// Column tiling of an n-wide GEMM: pick_bn's width for every tile.
void column_tiles(GemmParams &p, int64_t n, bool pair, bool a_mn)
{
    p.BN = pick_bn(n);
    p.num_n = (int)((n + p.BN - 1) / p.BN);
    p.idesc = idesc_bf16_f32(pair ? 2 * BM : BM, p.BN, a_mn, true);
}

// CTA pairs for 256-column tiles (each CTA then loads two whole 64-column boxes
// of B) when there is more than one 128-row block, unless switched off
// (CAAT_BWD_PAIR=0).  Narrower tiles stay on single CTAs: 128-column pair
// tiles run their MMAs at about half the rate per FLOP of 256-column ones, and
// 192-column tiles would split B into 96-column halves, which the 128-byte
// swizzle cannot lay out (the 64-byte one can, but measured no faster than
// single CTAs).
bool use_pairs(int64_t M, int64_t n)
{
    const char *env = std::getenv("CAAT_BWD_PAIR");
    if (env != nullptr && std::strcmp(env, "0") == 0) return false;
    return M > BM && pick_bn(n) == MAX_BN;
}

// Position of channel c in the order "the channels of S ascending, then the
// others ascending" (sel: the n_sel indices of S, ascending and unique): its rank
// in S, or n_sel plus the number of channels outside S below it.  A list that is
// not ascending can give a position outside [0, h): -1 then, and the callers skip
// the row.
__device__ __forceinline__ int64_t s_first_pos(const int32_t *__restrict__ sel, int64_t n_sel, int64_t h,
                                               int64_t c)
{
    int64_t lo = 0, hi = n_sel;                       // first i with sel[i] >= c
    while (lo < hi) {
        const int64_t mid = (lo + hi) >> 1;
        if ((int64_t)__ldg(sel + mid) < c) lo = mid + 1;
        else hi = mid;
    }
    const int64_t pos = (lo < n_sel && (int64_t)__ldg(sel + lo) == c) ? lo : n_sel + (c - lo);
    return (pos >= 0 && pos < h) ? pos : -1;
}

// fp32 [rows, cols] (row stride lds) -> bf16 (row stride ldd), 8 columns per
// thread.  With sel: destination row c takes source row s_first_pos(c) (the
// source rows in the S-first channel order, the destination in channel order).
__global__ void __launch_bounds__(256)
f32_rows_to_bf16_kernel(const float *__restrict__ src, int64_t rows, int64_t cols, int64_t lds,
                        uint16_t *__restrict__ dst, int64_t ldd, const int32_t *__restrict__ sel,
                        int64_t n_sel)
{
    const int64_t per_row = cols / 8;
    const int64_t total = rows * per_row;
    griddep_wait();                  // a programmatic dependent of the accumulating GEMM
    griddep_launch_dependents();
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t rr = i / per_row, c = (i - rr * per_row) * 8;
        const int64_t sr = sel != nullptr ? s_first_pos(sel, n_sel, rows, rr) : rr;
        if (sr < 0) continue;
        const float4 a = __ldcs(reinterpret_cast<const float4 *>(src + sr * lds + c));
        const float4 b = __ldcs(reinterpret_cast<const float4 *>(src + sr * lds + c + 4));
        const uint4 w = make_uint4(pack_bf16x2(__float_as_uint(a.x), __float_as_uint(a.y)),
                                   pack_bf16x2(__float_as_uint(a.z), __float_as_uint(a.w)),
                                   pack_bf16x2(__float_as_uint(b.x), __float_as_uint(b.y)),
                                   pack_bf16x2(__float_as_uint(b.z), __float_as_uint(b.w)));
        *reinterpret_cast<uint4 *>(dst + rr * ldd + c) = w;
    }
}

// Rows of a bf16 [h, K] matrix between channel order and the S-first order: with
// to_s_first, dst row s_first_pos(c) = src row c; else dst row c = src row
// s_first_pos(c).  One warp per row, 16-byte copies, eight in flight per lane.
// With room for it (dynamic shared memory of n_sel entries) S is staged in
// shared memory first, so that each row's binary search does not wait on a
// chain of global loads.
__global__ void __launch_bounds__(256)
permute_rows_kernel(const uint16_t *__restrict__ src, int64_t lds, uint16_t *__restrict__ dst, int64_t ldd,
                    int64_t h, int64_t K, const int32_t *__restrict__ sel, int64_t n_sel, int to_s_first,
                    int staged)
{
    extern __shared__ int32_t ssel[];
    // A programmatic dependent of the previous launch.  It does not let its own
    // dependent start early: that is the dX GEMM, whose persistent CTAs would sit
    // on every SM waiting for this short kernel and keep the dW GEMM (on the side
    // stream, which needs no permuted W) from running beside it.
    griddep_wait();
    if (staged) {
        for (int64_t i = threadIdx.x; i < n_sel; i += blockDim.x) ssel[i] = __ldg(sel + i);
        __syncthreads();
    }
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    const int64_t n16 = K / 8;
    for (int64_t c = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); c < h; c += warps) {
        int64_t pos = 0;
        if (lane == 0) {
            if (staged) {
                int64_t lo = 0, hi = n_sel;
                while (lo < hi) {
                    const int64_t mid = (lo + hi) >> 1;
                    if ((int64_t)ssel[mid] < c) lo = mid + 1;
                    else hi = mid;
                }
                pos = (lo < n_sel && (int64_t)ssel[lo] == c) ? lo : n_sel + (c - lo);
                if (pos < 0 || pos >= h) pos = -1;
            } else {
                pos = s_first_pos(sel, n_sel, h, c);
            }
        }
        pos = __shfl_sync(0xffffffffu, pos, 0);
        if (pos < 0) continue;                        // the whole warp
        const uint4 *s4 = reinterpret_cast<const uint4 *>(src + (to_s_first ? c : pos) * lds);
        uint4 *d4 = reinterpret_cast<uint4 *>(dst + (to_s_first ? pos : c) * ldd);
        int64_t i = lane;
        for (; i + 224 < n16; i += 256) {
            uint4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) v[u] = __ldcs(s4 + i + 32 * u);
#pragma unroll
            for (int u = 0; u < 8; ++u) d4[i + 32 * u] = v[u];
        }
        for (; i < n16; i += 32) d4[i] = __ldcs(s4 + i);
    }
}

// Split of the K range into k parts of ceil(nkb / k) k-blocks (every part
// non-empty); units = tiles * parts.
void set_ksplit(GemmParams &p, int k, int tiles)
{
    p.kbps = (p.nkb + k - 1) / k;
    p.ksplit = (p.nkb + p.kbps - 1) / p.kbps;
    p.units = tiles * p.ksplit;
}

// The split (1..8 parts, at least 8 k-blocks per part) with the fewest
// waves-of-work over `slots` workers, per part
void pick_ksplit(GemmParams &p, int tiles, int slots)
{
    // Each extra part adds an fp32 reduce-add of the whole of dW.  Only tiles
    // that do not fill one round of the slots are split (at the 1.1B
    // down-projection, 192 pair tiles on 76 pairs, a 7-way split added about
    // 320 MB of reduce traffic and cost 35 us), and each extra part is charged
    // 0.05 rounds: the 130M down-projection (96 tiles on 152 SMs) still splits
    // three ways (2 rounds / 3 + 0.1 < 1; 3.5 us faster), the 1.1B out-projection
    // (64 pair tiles on 76 pairs) no longer seven ways (6 rounds / 7 + 0.3 > 1;
    // that split cost 15 us).
    if (tiles >= slots) {
        set_ksplit(p, 1, tiles);
        return;
    }
    int best = 1;
    double best_cost = (double)((tiles + slots - 1) / slots);
    for (int k = 2; k <= 8 && p.nkb / k >= 8; ++k) {
        const double cost = (double)((tiles * k + slots - 1) / slots) / k + 0.05 * (k - 1);
        if (cost < best_cost - 1e-9) { best = k; best_cost = cost; }
    }
    set_ksplit(p, best, tiles);
}

}  // namespace

namespace {
thread_local SideStream t_side[64];
}  // namespace

// A second stream per host thread and device, with a fork and a join event: the
// dW chain of the backward runs on it next to dX (they only read shared inputs),
// so dW's CTAs take SMs as soon as dX's retire instead of after dX has drained.
// Created on first use outside stream capture; per thread, so that concurrent
// callers never interleave their fork/join events.  "CAAT_BWD_SIDE_STREAM=0"
// (or no stream could be made) gives null: everything stays on `main`.

SideStream *side_stream(cudaStream_t main)
{
    const char *env = std::getenv("CAAT_BWD_SIDE_STREAM");
    if (env != nullptr && std::strcmp(env, "0") == 0) return nullptr;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    SideStream &sd = t_side[dev];
    if (sd.s == nullptr) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(main, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) return nullptr;
        cudaStream_t s2 = nullptr;
        cudaEvent_t f = nullptr, j = nullptr;
        if (cudaStreamCreateWithFlags(&s2, cudaStreamNonBlocking) != cudaSuccess) return nullptr;
        if (cudaEventCreateWithFlags(&f, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&j, cudaEventDisableTiming) != cudaSuccess) {
            if (f) cudaEventDestroy(f);
            cudaStreamDestroy(s2);
            return nullptr;
        }
        sd.s = s2;
        sd.fork = f;
        sd.join = j;
    }
    return &sd;
}

bool bwd_tc_supported(int t, int64_t N, int64_t K, int64_t h, const void *X, int64_t ldx,
                      const void *W, int64_t ldw, const ConstPtrs &dY, int64_t ld_dy, const void *dX,
                      int64_t lddx, const void *dW, int64_t ld_dw)
{
    const int64_t kt = K / t;
    if (t > MAX_T_TC || kt < 64 || kt % 8 != 0 || N < BM || h < 256 || h % 8 != 0) return false;
    if (N > (int64_t)INT32_MAX || h > (int64_t)INT32_MAX) return false;
    if (ldx % 8 || ldw % 8 || ld_dy % 8 || lddx % 8 || ld_dw % 8) return false;
    if ((uintptr_t)X % 16 || (uintptr_t)W % 16 || (uintptr_t)dX % 16 || (uintptr_t)dW % 16) return false;
    for (int r = 0; r < t; ++r)
        if ((uintptr_t)dY.p[r] % 16) return false;
    return true;
}

// dX[:, shard r] = dY_r W_r^T and dW[shard r, :] = X_r^T dY_r for every rank.
// W and dW are in the nn.Linear layout ([h, K] storage, row stride ldw / ld_dw).
// A null dX or dW skips that product (the column-parallel layer uses one at a time).
caat_status launch_rowpar_bwd_tc(int t, int64_t N, int64_t K, int64_t h, const void *X, int64_t ldx,
                                 const void *W, int64_t ldw, const ConstPtrs &dY, int64_t ld_dy,
                                 void *dX, int64_t lddx, void *dW, int64_t ld_dw, float *wacc,
                                 int64_t s_sum, const void *dsum, int64_t ld_dsum, cudaStream_t s,
                                 bool own_compact, const int32_t *row_sel, int64_t row_nsel, void *dw_tmp,
                                 void *w_perm)
{
    const int64_t kt = K / t;
    if (s_sum < 0 || s_sum > h || s_sum % 64 != 0 || (s_sum > 0 && dsum == nullptr)) return CAAT_ERR_UNSUPPORTED;
    if (row_sel != nullptr && dW != nullptr && (dw_tmp == nullptr || (uintptr_t)dw_tmp % 16 != 0 || K % 8 != 0))
        return CAAT_ERR_UNSUPPORTED;
    const int64_t h_own = h - s_sum;           // channels read from each rank's own gradient

    // A-operand maps: rank r's gradient from channel s_sum on (each rank; in the
    // compact form its columns start there), and the reduced sum of channels
    // [0, s_sum) (box shapes differ between dX and dW)
    auto grad_maps = [&](TmapArray &am, CUtensorMap &sm, uint32_t box0, uint32_t box1) -> bool {
        for (int r = 0; r < t; ++r) {
            if (h_own == 0) { am.m[r] = CUtensorMap{}; continue; }
            const uint64_t dims[2] = {(uint64_t)h_own, (uint64_t)N};
            const uint64_t str[1] = {(uint64_t)ld_dy * 2};
            const uint32_t box[2] = {box0, box1};
            const uint16_t *own = (const uint16_t *)dY.p[r] + (own_compact ? 0 : s_sum);
            if (!encode_tmap(&am.m[r], own, 2, dims, str, box)) return false;
        }
        if (s_sum == 0) { sm = am.m[0]; return true; }
        const uint64_t dims[2] = {(uint64_t)s_sum, (uint64_t)N};
        const uint64_t str[1] = {(uint64_t)ld_dsum * 2};
        const uint32_t box[2] = {box0, box1};
        return encode_tmap(&sm, dsum, 2, dims, str, box);
    };

    // dW on the side stream when both products are wanted
    cudaStream_t sw = s;
    SideStream *side = (dX != nullptr && dW != nullptr) ? side_stream(s) : nullptr;
    if (side != nullptr) {
        if (cudaEventRecord(side->fork, s) != cudaSuccess || cudaStreamWaitEvent(side->s, side->fork, 0) != cudaSuccess)
            return CAAT_ERR_CUDA;
        sw = side->s;
    }
    auto join = [&](caat_status st) -> caat_status {
        if (side == nullptr) return st;
        if (cudaEventRecord(side->join, sw) != cudaSuccess || cudaStreamWaitEvent(s, side->join, 0) != cudaSuccess)
            return CAAT_ERR_CUDA;
        return st;
    };
    // ---- dX = dY_r W_r^T: A = dY_r (K-major), B = W_r^T (MN-major)
    if (dX != nullptr) {
        if (w_perm != nullptr) {
            // W's rows in the S-first order (the order of dY's channels) first; the
            // dW chain, on the side stream, does not read W and runs beside it
            const caat_status st = launch_permute_rows(W, ldw, w_perm, K, h, K, row_sel, row_nsel, true, s);
            if (st != CAAT_OK) return join(st);
            W = w_perm;
            ldw = K;
        }
        TmapArray am;
        CUtensorMap sm;
        if (!grad_maps(am, sm, 64, BM)) return CAAT_ERR_UNSUPPORTED;
        const bool pair = use_pairs(N, kt);
        CUtensorMap bm;
        const uint64_t dims[3] = {(uint64_t)kt, (uint64_t)t, (uint64_t)h};
        const uint64_t str[2] = {(uint64_t)kt * 2, (uint64_t)ldw * 2};
        const uint32_t box[3] = {64, 1, 64};
        if (!encode_tmap(&bm, W, 3, dims, str, box)) return CAAT_ERR_UNSUPPORTED;
        GemmParams p{};
        p.M = N; p.Nn = kt; p.Kk = h;
        p.t = t;
        p.num_m = (int)((N + BM - 1) / BM);
        column_tiles(p, kt, pair, false);
        p.nkb = (int)((h + BK - 1) / BK);
        p.s_blocks = (int)(s_sum / 64);
        set_ksplit(p, 1, t * (pair ? (p.num_m + 1) / 2 : p.num_m) * p.num_n);
        CUtensorMap cm;
        const uint64_t cdims[3] = {(uint64_t)kt, (uint64_t)t, (uint64_t)N};
        const uint64_t cstr[2] = {(uint64_t)kt * 2, (uint64_t)lddx * 2};
        const uint32_t cbox[3] = {64, 1, 32};
        if (!encode_tmap(&cm, dX, 3, cdims, cstr, cbox)) return CAAT_ERR_UNSUPPORTED;
        const caat_status st = pair ? launch_grouped<false, false, true>(am, sm, bm, cm, p, s, "rowpar_bwd_dx_tc")
                                    : launch_grouped<false, false, false>(am, sm, bm, cm, p, s, "rowpar_bwd_dx_tc");
        if (st != CAAT_OK) return st;
    }
    if (dW == nullptr) return CAAT_OK;
    // ---- dW^T = dY_r^T X_r: A = dY_r^T (MN-major), B = X_r (MN-major)
    auto dw_chain = [&]() -> caat_status {
        TmapArray am;
        CUtensorMap sm;
        if (!grad_maps(am, sm, 64, 64)) return CAAT_ERR_UNSUPPORTED;
        const bool pair = use_pairs(h, kt);
        CUtensorMap bm;
        const uint64_t dims[3] = {(uint64_t)kt, (uint64_t)t, (uint64_t)N};
        const uint64_t str[2] = {(uint64_t)kt * 2, (uint64_t)ldx * 2};
        const uint32_t box[3] = {64, 1, 64};
        if (!encode_tmap(&bm, X, 3, dims, str, box)) return CAAT_ERR_UNSUPPORTED;
        GemmParams p{};
        p.M = h; p.Nn = kt; p.Kk = N;
        p.t = t;
        p.num_m = (int)((h + BM - 1) / BM);
        column_tiles(p, kt, pair, true);
        p.nkb = (int)((N + BK - 1) / BK);
        p.s_blocks = (int)(s_sum / 64);
        const int tiles = t * (pair ? (p.num_m + 1) / 2 : p.num_m) * p.num_n;
        if (wacc != nullptr) pick_ksplit(p, tiles, pair ? num_sms() / 2 : num_sms());
        else set_ksplit(p, 1, tiles);
        if (p.ksplit == 1) {
            // straight to dW; with row_sel to dw_tmp [h, K] in the S-first row
            // order, then rows back to channel order
            void *dst = row_sel != nullptr ? dw_tmp : dW;
            const int64_t ldd = row_sel != nullptr ? K : ld_dw;
            CUtensorMap cm;
            const uint64_t cdims[3] = {(uint64_t)kt, (uint64_t)t, (uint64_t)h};
            const uint64_t cstr[2] = {(uint64_t)kt * 2, (uint64_t)ldd * 2};
            const uint32_t cbox[3] = {64, 1, 32};
            if (!encode_tmap(&cm, dst, 3, cdims, cstr, cbox)) return CAAT_ERR_UNSUPPORTED;
            caat_status st = pair ? launch_grouped<true, false, true>(am, sm, bm, cm, p, sw, "rowpar_bwd_dw_tc")
                                  : launch_grouped<true, false, false>(am, sm, bm, cm, p, sw, "rowpar_bwd_dw_tc");
            if (st != CAAT_OK || row_sel == nullptr) return st;
            return launch_permute_rows((const uint16_t *)dw_tmp, K, dW, ld_dw, h, K, row_sel, row_nsel, false, sw);
        }
        // split over tokens: fp32 partials reduce-added into wacc [h, K], then one
        // rounding to bf16 into dW (with row_sel: rows back in channel order)
        CUtensorMap cm;
        const uint64_t cdims[3] = {(uint64_t)kt, (uint64_t)t, (uint64_t)h};
        const uint64_t cstr[2] = {(uint64_t)kt * 4, (uint64_t)K * 4};
        const uint32_t cbox[3] = {32, 1, 32};
        if (!encode_tmap(&cm, wacc, 3, cdims, cstr, cbox, true)) return CAAT_ERR_UNSUPPORTED;
        if (cudaMemsetAsync(wacc, 0, (size_t)h * (size_t)K * 4, sw) != cudaSuccess) return CAAT_ERR_CUDA;
        caat_status st = pair ? launch_grouped<true, true, true>(am, sm, bm, cm, p, sw, "rowpar_bwd_dw_tc")
                              : launch_grouped<true, true, false>(am, sm, bm, cm, p, sw, "rowpar_bwd_dw_tc");
        if (st != CAAT_OK) return st;
        const int64_t total = h * (K / 8);
        int64_t blocks = (total + 255) / 256;
        if (blocks > (int64_t)num_sms() * 8) blocks = (int64_t)num_sms() * 8;
        launch_dependent(f32_rows_to_bf16_kernel, dim3((unsigned)blocks), dim3(256), 0, sw, (const float *)wacc, h,
                         K, K, (uint16_t *)dW, ld_dw, row_sel, row_nsel);
        note_launch("rowpar_bwd_dw_tc", 1);
        return cudaGetLastError() == cudaSuccess ? CAAT_OK : CAAT_ERR_CUDA;
    };
    return join(dw_chain());
}

caat_status launch_permute_rows(const void *src, int64_t lds, void *dst, int64_t ldd, int64_t h, int64_t K,
                                const int32_t *sel, int64_t n_sel, bool to_s_first, cudaStream_t s)
{
    if (h == 0 || K == 0) return CAAT_OK;
    if (K % 8 != 0 || lds % 8 != 0 || ldd % 8 != 0 || (uintptr_t)src % 16 != 0 || (uintptr_t)dst % 16 != 0)
        return CAAT_ERR_UNSUPPORTED;
    int64_t blocks = (h + 7) / 8;                     // 8 warps per CTA, one row per warp
    if (blocks > (int64_t)num_sms() * 8) blocks = (int64_t)num_sms() * 8;
    const bool staged = n_sel <= 8192;                // up to 32 KB of shared memory
    const size_t smem = staged ? (size_t)n_sel * 4 : 0;
    launch_dependent(permute_rows_kernel, dim3((unsigned)blocks), dim3(256), smem, s, (const uint16_t *)src, lds,
                     (uint16_t *)dst, ldd, h, K, sel, n_sel, to_s_first ? 1 : 0, staged ? 1 : 0);
    note_launch("permute_rows", 1);
    return cudaGetLastError() == cudaSuccess ? CAAT_OK : CAAT_ERR_CUDA;
}

}  // namespace caat
