// kda_bwd_tc.cu -- bf16 path of kda_chunk_bwd_varlen (d_qk = d_v = 128): the gradients of the
// chunked KDA forward on tcgen05 tensor cores.
//
// Method: [RFC-0026] "RFC-0026: Ling3 KDA Varlen 支持（packing 文档间隔离）", 背景 "KDA 状态泄漏问题"
// (S_t = S_{t-1} exp(g_t) + beta_t k_t v_t^T with rows = key channels, o_t = scale S_t^T q_t) and
// §3.1.1 (S = 0 at every segment start, id 0 = padding). The pages state the forward only; the
// backward is its derivative (the same equations as the fp32 walks of kda_bwd.cu), organised by
// 64-token chunks:
//
//   per chunk c and head: S_in = the state its carried segment brings in (row = key channel),
//   D_end = dL/dS at the chunk's last token for the segment that goes on into chunk c + 1.
//   Within the chunk (tokens t, s; Suf_t = sum of g over the chunk's real tokens after t;
//   Qt_t = q_t exp(-Suf_t), Ktb_s = beta_s k_s exp(Suf_s), as in the forward kernel):
//     M_ts  = 1 when t is real and s lies in t's segment with s <= t
//     A'    = scale * M . (Qt Ktb^T)          W = M . (dO V^T)
//     dq_t  = scale exp(-Suf_t) [ (W Ktb)_t + [t carried] S_dec do_t ],   S_dec = diag(P) S_in
//     dk_s  = beta_s exp(Suf_s) [ scale (W^T Qt)_s + [s in the last segment] D_end v_s ]
//     dv_s  = (A'^T dO)_s + [s in the last segment] D_end^T Ktb_s
//     dbeta_s = k_s . (dk_s / beta_s)
//     dg_t  = sum over u >= t of t's segment within the chunk of (q_u dq_u - k_u dk_u)
//             + [t in the last segment] sum_j S_out[i][j] D_end[i][j]      (per channel i)
//   where P = exp(sum of the chunk's real g), S_out = the state at the chunk's end; dg is 0 at a
//   segment's first token (g_t there multiplies a zero state).
//   The last line is the identity dL/dG_u = q_u dq_u - k_u dk_u (o depends on the cumulative
//   log-decay G only through G_t - G_s), summed over the tokens whose G g_t enters; the part
//   past the chunk is the direct form of dg at the next chunk's first token.
//
// After a small planner (which also cuts chains longer than 32 chunks into 16-chunk pieces,
// each scan then running as an end-state pass, a combine pass and the export pass), three
// kernels, and a last one that is empty unless needed:
//   scan_kernel<false>  walks each chain of chunks that one segment links (a chunk holding a
//     start or padding begins a chain) forward in time and stores S_in of every chunk:
//     S^T (+)= V^T Khat with Khat = beta k exp(Suf) on the rows that reach the chunk's end.
//   scan_kernel<true>   walks the same chains backward and stores D_end:
//     D^T = D^T diag(P) + dO^T Qhat, Qhat_t = scale q_t exp(G_t) on the rows of the segment the
//     chunk carries in (G_t = sum of g over the chunk's first t + 1 tokens).
//   grad_kernel         one (chunk, head) at a time, all gradients (eight MMAs, below).
//   redo_kernel         the items the gradient kernel listed, in fp32 (below).
// The scans keep the state in tensor memory (fp32) and export it per chunk; the exponentials
// there stay within (0, 1], so they need no range check. The gradient kernel's factors
// exp(-Suf) and exp(Suf) do: a chunk whose log-decay on some channel falls below -80 is
// listed, and redo_kernel rewrites its gradients by the token recurrence over the chunk,
// from the stored S_in and D_end.
//
// Precision: as in the forward kernel, Qt, Ktb, A' and W are carried as hi + lo bf16 pairs and
// each product sums the pairs' cross terms; dO and V enter exactly. S_in and D_end are hi + lo
// pairs too: rounded once to bf16 (as the forward rounds its S_dec), S_in alone puts dq's worst
// error at 1.24x the bound on a chunk between two carried ones (fp64 emulation), D_end dk's at
// 0.6x. Accumulation is fp32 in tensor memory.
//
// Gradient-kernel tensor-core mapping (kind::f16, transposed outputs: lane = channel, column =
// token, so that the epilogue's suffix sum over tokens runs within a thread). Qt carries the
// factor scale here (so SC, A' and the dK product include it):
//   SC    = Qt Ktb^T          M=64  N=64 K=128  A, B K-major                     x3
//   W     = dO V^T            M=64  N=64 K=128  A, B K-major                     x1
//   Qs^T  = S_in dO^T         M=128 N=64 K=128  A K-major (128 rows), B K-major  x2  -> QQ
//   T2^T  = D_end V^T         M=128 N=64 K=128  A K-major (128 rows), B K-major  x2  -> KK
//   Vs^T  = D_end^T Ktb^T     M=128 N=64 K=128  A MN-major, B K-major            x3  -> VV
//   then the prologue warps scale QQ by P and keep its carried rows, and keep the last
//   segment's rows of KK and VV, in tensor memory, and the last three accumulate onto them:
//   dQ^T += Ktb^T W^T         M=128 N=64 K=64   A MN-major, B K-major            x3  -> QQ
//   dK^T += Qt^T W            M=128 N=64 K=64   A MN-major, B MN-major           x3  -> KK
//   dV^T += dO^T A'           M=128 N=64 K=64   A MN-major, B MN-major           x2  -> VV
// QQ, KK and VV are double-buffered, so that an item's products run during the previous item's
// epilogue.
// Warp roles (320 threads): 0 TMA producer, 1 MMA issuer, 2-5 prologue (one key channel per
// thread: Suf, Qt and Ktb), 6-9 the states' conversion, the A' and W tiles and the epilogue.
// Shared memory holds one item (224 KB of tiles); the lo halves of S_dec and D_end borrow the
// k and g tiles (free once the prologue has read them; the epilogue reads k and g from L2) and
// the A' and W tiles (written only after the products that read D_end_lo have completed).
#include "kda_common.cuh"
#include "kda_plan.cuh"
#include "kda_sm100.cuh"

namespace kda {
namespace tc {
bool make_map(CUtensorMap* map, const void* base, int64_t N, int32_t H);   // kda_chunk_tc.cu
}

namespace tcb {

using namespace kda::sm100;
using tc::ChunkMeta;
using tc::align256;

constexpr int D = 128;
constexpr int C = kChunk;
constexpr uint32_t kTile = C * D * 2;        // 16 KB: 64 rows x 128 bf16, two 8 KB panels
constexpr uint32_t kPanel = kTile / 2;
constexpr uint32_t kTile128 = D * D * 2;     // 32 KB: 128 rows x 128 bf16, two 16 KB panels
constexpr uint32_t kPanel128 = kTile128 / 2;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRangeLog2 = -80.f * kLog2e;  // a chunk's log-decay below -80, in base 2
constexpr size_t kStateBytes = size_t(D) * D * 4;

// ---- workspace ------------------------------------------------------------------------

// A chain longer than kPiece chunks is cut into pieces of kPiece chunks (in the scan's own
// order), which run at once: a first pass leaves each piece's end state from a zero start and
// the product of its chunks' decays in a slot, a combine pass turns those into every piece's
// true start state, and the export pass starts each piece from it.
constexpr int kPiece = 16;

__host__ __device__ inline int64_t max_pieces(int64_t n_chunks) { return 2 * n_chunks + 8; }
__host__ __device__ inline int64_t max_slots(int64_t n_chunks) {
    return 2 * ((n_chunks + kPiece - 1) / kPiece) + 8;
}
constexpr size_t kSlotBytes = size_t(128) * 128 * 4 + 512;   // fp32 state + decay product

struct BDir {                      // one scan direction's work lists
    int4* pieces;                  // (chain, piece number, pieces in the chain, first slot or -1)
    int32_t* order;                // pieces, longest first
    int32_t* pieces_a;             // pieces that leave an end state (all but a chain's last)
    int4* split;                   // chains cut into pieces: (chain, pieces, first slot, 0)
    uint8_t* slots;                // [slots][H] kSlotBytes each
};

struct BPlan {
    int32_t* counters;     // [0] chains, [1]/[2] next export-pass item (forward/reverse), [3]
                           // items the gradient kernel left to the fp32 redo, [4]/[5] pieces,
                           // [6]/[7] pieces with an end state, [8]/[9] chains cut into pieces,
                           // [10]/[11] next end-state item, [12]/[13] next combine item
    ChunkMeta* meta;       // [n_chunks] start / real-token masks
    int32_t* first_cut;    // [n_chunks] first start-or-padding row, 64 if none
    int2* chains;          // [n_chunks] (first chunk, chunk after the last)
    int32_t* redo_flag;    // [n_chunks * H] 1 once the (chunk, head) item is listed in redo
    int32_t* redo;         // [n_chunks * H] items outside the factorised form's range
    BDir dir[2];           // forward, reverse
    float* s_in;           // [n_chunks][H] state entering the chunk, as hi and lo bf16 tiles
    float* d_end;          // [n_chunks][H] adjoint at the chunk's end, likewise (each 2 x 32 KB:
                           // 128 x 128, row = key channel, K-major 128B-swizzled)
};

__host__ __device__ inline size_t bdir_bytes(int64_t n_chunks, int32_t H) {
    const size_t np = size_t(max_pieces(n_chunks));
    return align256(np * 16) + align256(np * 4) * 2 + align256(size_t(n_chunks) * 16) +
           size_t(max_slots(n_chunks)) * H * kSlotBytes;
}

__host__ __device__ inline size_t bplan_bytes(int64_t n_chunks, int32_t H) {
    return align256(64 * 4) + align256(size_t(n_chunks) * sizeof(ChunkMeta)) +
           align256(size_t(n_chunks) * 4) + align256(size_t(n_chunks) * 8) +
           align256(size_t(n_chunks) * H * 4) * 2 + 2 * align256(bdir_bytes(n_chunks, H));
}

__host__ __device__ inline BPlan bplan_view(void* ws, int64_t n_chunks, int32_t H) {
    uint8_t* p = static_cast<uint8_t*>(ws);
    BPlan pl;
    pl.counters = reinterpret_cast<int32_t*>(p);   p += align256(64 * 4);
    pl.meta = reinterpret_cast<ChunkMeta*>(p);     p += align256(size_t(n_chunks) * sizeof(ChunkMeta));
    pl.first_cut = reinterpret_cast<int32_t*>(p);  p += align256(size_t(n_chunks) * 4);
    pl.chains = reinterpret_cast<int2*>(p);        p += align256(size_t(n_chunks) * 8);
    pl.redo_flag = reinterpret_cast<int32_t*>(p);  p += align256(size_t(n_chunks) * H * 4);
    pl.redo = reinterpret_cast<int32_t*>(p);       p += align256(size_t(n_chunks) * H * 4);
    for (int d = 0; d < 2; ++d) {
        uint8_t* q = p;
        const size_t np = size_t(max_pieces(n_chunks));
        pl.dir[d].pieces = reinterpret_cast<int4*>(q);  q += align256(np * 16);
        pl.dir[d].order = reinterpret_cast<int32_t*>(q); q += align256(np * 4);
        pl.dir[d].pieces_a = reinterpret_cast<int32_t*>(q); q += align256(np * 4);
        pl.dir[d].split = reinterpret_cast<int4*>(q);   q += align256(size_t(n_chunks) * 16);
        pl.dir[d].slots = q;
        p += align256(bdir_bytes(n_chunks, H));
    }
    pl.s_in = reinterpret_cast<float*>(p);         p += size_t(n_chunks) * H * kStateBytes;
    pl.d_end = reinterpret_cast<float*>(p);
    return pl;
}

// ---- small device helpers -------------------------------------------------------------

// Byte offset of element (r, ch) of a 64-row x 128-column K-major 128B-swizzled tile.
__device__ __forceinline__ uint32_t eoff(int r, int ch) {
    return (ch >> 6) * kPanel + r * 128 + ((((ch >> 3) & 7) ^ (r & 7)) << 4) + (ch & 7) * 2;
}
// ... of a 128-row x 128-column tile (two 16 KB panels of 128-byte rows).
__device__ __forceinline__ uint32_t eoff128(int r, int ch) {
    return (ch >> 6) * kPanel128 + r * 128 + ((((ch >> 3) & 7) ^ (r & 7)) << 4) + (ch & 7) * 2;
}

__device__ __forceinline__ float ld_bf(const uint8_t* base, uint32_t off) {
    return __uint_as_float(uint32_t(*reinterpret_cast<const uint16_t*>(base + off)) << 16);
}
__device__ __forceinline__ uint32_t ld32(const uint8_t* base, uint32_t off) {
    return *reinterpret_cast<const uint32_t*>(base + off);
}
__device__ __forceinline__ void st32(uint8_t* base, uint32_t off, uint32_t v) {
    *reinterpret_cast<uint32_t*>(base + off) = v;
}
// bf16 pair (even element in the low half) -> fp32 pair, exactly
__device__ __forceinline__ float2 unpk2(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
// packed fp32 pair arithmetic (one f32x2 instruction for two lanes of work)
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 u, v, w;\n\tmov.b64 u, {%2, %3};\n\tmov.b64 v, {%4, %5};\n\t"
        "mul.rn.f32x2 w, u, v;\n\tmov.b64 {%0, %1}, w;\n\t}"
        : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 u, v, w;\n\tmov.b64 u, {%2, %3};\n\tmov.b64 v, {%4, %5};\n\t"
        "add.rn.f32x2 w, u, v;\n\tmov.b64 {%0, %1}, w;\n\t}"
        : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 u, v, w, z;\n\tmov.b64 u, {%2, %3};\n\tmov.b64 v, {%4, %5};\n\t"
        "mov.b64 w, {%6, %7};\n\tfma.rn.f32x2 z, u, v, w;\n\tmov.b64 {%0, %1}, z;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}
// (a, b) -> a bf16 pair, a in the low half; round to nearest even
__device__ __forceinline__ uint32_t pack2(float a, float b) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
}
// (a, b) = hi + lo as bf16 pairs: hi = bf16 of each, lo = bf16 of the remainder
__device__ __forceinline__ void split2(float a, float b, uint32_t& hi, uint32_t& lo) {
    hi = pack2(a, b);
    lo = pack2(a - __uint_as_float(hi << 16), b - __uint_as_float(hi & 0xffff0000u));
}
// 2^x on the multi-function unit (ex2.approx: within 2 ulp)
__device__ __forceinline__ float ex2a(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity) {
    const bool ok = mbar_wait(bar, parity);
    return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void set_status(uint32_t* status, uint32_t bit) {
    if (status) atomicOr(status, bit);
}

// 32x32b shape, 8 consecutive columns.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
}

// 32x32b shape, 8 consecutive columns, registers to tensor memory.
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
                 ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]),
                   "r"(r[6]), "r"(r[7])
                 : "memory");
}

// A barrier among four warps on an mbarrier of count 4 (bounded like every other wait: a
// warp that gave up elsewhere cannot leave the others waiting for ever). `uses` counts the
// warp's previous passes, whose parity the wait needs. Returns false on a timeout.
__device__ __forceinline__ bool group_sync(uint64_t* bar, uint32_t& uses, int lane) {
    __syncwarp();
    if (lane == 0) mbar_arrive(bar);
    const bool ok = warp_wait(bar, uses & 1);
    ++uses;
    return ok;
}

// Rows s of t's segment with s <= t (bit s), none when t is padding.
__device__ __forceinline__ unsigned long long keep_bits(unsigned long long start,
                                                        unsigned long long valid, int t) {
    if (!((valid >> t) & 1ull)) return 0ull;
    const unsigned long long upto = (t == 63) ? ~0ull : ((2ull << t) - 1ull);
    const unsigned long long st = start & upto;
    const int lo = st ? 63 - __clzll((long long)st) : 0;
    return upto & (~0ull << lo);
}

// K-major descriptor offsets (in 16-byte units) of K step kk (16 elements) of a 128-wide K:
// 32 bytes within a 128-byte row, then the next panel.
__device__ __forceinline__ uint64_t kofs64(int kk) {
    return uint64_t(((kk >> 2) * kPanel + (kk & 3) * 32) >> 4);
}
__device__ __forceinline__ uint64_t kofs128(int kk) {
    return uint64_t(((kk >> 2) * kPanel128 + (kk & 3) * 32) >> 4);
}

// ---- planner ----------------------------------------------------------------------------

// Per chunk: the start and real-token masks (one warp per chunk, ballots) and the first
// start-or-padding row.
__global__ void __launch_bounds__(256)
bwd_masks_kernel(const int32_t* __restrict__ seg, int64_t N, RowStartTest row_start,
                 int64_t n_chunks, int32_t H, void* ws) {
    BPlan pl = bplan_view(ws, n_chunks, H);
    const int lane = threadIdx.x & 31;
    const int64_t c = int64_t(blockIdx.x) * 8 + (threadIdx.x >> 5);
    if (c >= n_chunks) return;
    bool st[2], va[2];
#pragma unroll
    for (int hlf = 0; hlf < 2; ++hlf) {
        const int64_t p = c * C + hlf * 32 + lane;
        va[hlf] = p < N && is_real(seg, p);
        st[hlf] = va[hlf] && is_segment_start(seg, p, row_start);
    }
    const unsigned long long sm = (unsigned long long)__ballot_sync(0xffffffffu, st[0]) |
                                  ((unsigned long long)__ballot_sync(0xffffffffu, st[1]) << 32);
    const unsigned long long vm = (unsigned long long)__ballot_sync(0xffffffffu, va[0]) |
                                  ((unsigned long long)__ballot_sync(0xffffffffu, va[1]) << 32);
    if (lane == 0) {
        pl.meta[c].start = sm;
        pl.meta[c].valid = vm;
        const unsigned long long cut = sm | ~vm;
        pl.first_cut[c] = cut ? (__ffsll((long long)cut) - 1) : C;
    }
    for (int h = lane; h < H; h += 32) pl.redo_flag[c * H + h] = 0;
}

constexpr int kChainThreads = 1024;

__device__ int chain_scan(int v, int* s_warp, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int w = s_warp[lane];
        int wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += n;
        }
        s_warp[lane] = wi - w;
        if (lane == 31) *total = wi;
    }
    __syncthreads();
    const int r = s_warp[warp] + incl - v;
    __syncthreads();
    return r;
}

// Chains: a chain begins at chunk 0 and at every chunk holding a start or padding, and ends
// before the next such chunk; no state crosses a chain's first chunk's last cut backwards or
// its end forwards except through the chunk that ends it. Each scan direction's chains become
// pieces, ordered longest first (a counting sort on lengths 1 .. kPiece). One CTA.
__global__ void __launch_bounds__(kChainThreads, 1)
bwd_chains_kernel(int64_t n_chunks, int32_t H, int32_t split_min, void* ws) {
    BPlan pl = bplan_view(ws, n_chunks, H);
    __shared__ int s_warp[32];
    __shared__ int s_total;
    __shared__ int hist[kChainThreads];
    const int tid = threadIdx.x;
    int base = 0;
    for (int64_t c0 = 0; c0 < n_chunks; c0 += kChainThreads) {
        const int64_t c = c0 + tid;
        const int flag = (c < n_chunks && (c == 0 || pl.first_cut[c] < C)) ? 1 : 0;
        const int off = chain_scan(flag, s_warp, &s_total);
        if (flag) pl.chains[base + off].x = int(c);
        base += s_total;
        __syncthreads();
    }
    const int n = base;
    for (int k = tid; k < n; k += kChainThreads)
        pl.chains[k].y = (k + 1 < n) ? pl.chains[k + 1].x : int(n_chunks);
    __syncthreads();
    // Pieces, per scan direction. The forward scan runs chunks c_a .. c_b - 1; the reverse one
    // runs c_from down to c_a + 1, where c_from = c_b when the chain's end chunk carries rows
    // of its segment (first cut > 0), else c_b - 1. A run of L chunks is one piece when
    // L <= kPiece, else ceil(L / kPiece) pieces, each but the last with a slot.
    for (int d = 0; d < 2; ++d) {
        BDir& bd = pl.dir[d];
        int p_base = 0, a_base = 0, s_base = 0, x_base = 0;
        for (int k0 = 0; k0 < n; k0 += kChainThreads) {
            const int k = k0 + tid;
            int len = 0;
            if (k < n) {
                const int2 ch = pl.chains[k];
                if (d == 0) {
                    len = ch.y - ch.x;
                } else {
                    const bool head = ch.y < n_chunks && pl.first_cut[ch.y] > 0;
                    len = (head ? ch.y : ch.y - 1) - ch.x;
                }
            }
            const int np = len <= 0 ? 0 : (len <= split_min ? 1 : (len + kPiece - 1) / kPiece);
            const int cut = np > 1 ? 1 : 0;
            const int p_off = chain_scan(np, s_warp, &s_total);
            const int p_tot = s_total;
            const int a_off = chain_scan(cut ? np - 1 : 0, s_warp, &s_total);
            const int a_tot = s_total;
            const int x_off = chain_scan(cut, s_warp, &s_total);
            const int x_tot = s_total;
            const int slot = s_base + a_off;           // one slot per piece but the last
            for (int j = 0; j < np; ++j) {
                bd.pieces[p_base + p_off + j] = make_int4(k, j, np, cut ? slot : -1);
                if (cut && j < np - 1) bd.pieces_a[a_base + a_off + j] = p_base + p_off + j;
            }
            if (cut) bd.split[x_base + x_off] = make_int4(k, np, slot, 0);
            p_base += p_tot;
            a_base += a_tot;
            s_base += a_tot;
            x_base += x_tot;
            __syncthreads();
        }
        // pieces longest first (lengths 1 .. kPiece)
        auto plen = [&](int i) {
            const int4 pc = bd.pieces[i];
            const int2 ch = pl.chains[pc.x];
            int len;
            if (d == 0) {
                len = ch.y - ch.x;
            } else {
                const bool head = ch.y < n_chunks && pl.first_cut[ch.y] > 0;
                len = (head ? ch.y : ch.y - 1) - ch.x;
            }
            return pc.z == 1 ? min(len, kPiece) : min(kPiece, len - pc.y * kPiece);
        };
        if (tid <= kPiece) hist[tid] = 0;
        __syncthreads();
        for (int i = tid; i < p_base; i += kChainThreads) atomicAdd(&hist[kPiece - plen(i)], 1);
        __syncthreads();
        if (tid == 0) {
            int run = 0;
            for (int b = 0; b <= kPiece; ++b) {
                const int c = hist[b];
                hist[b] = run;
                run += c;
            }
        }
        __syncthreads();
        for (int i = tid; i < p_base; i += kChainThreads)
            bd.order[atomicAdd(&hist[kPiece - plen(i)], 1)] = i;
        __syncthreads();
        if (tid == 0) {
            pl.counters[4 + d] = p_base;
            pl.counters[6 + d] = a_base;
            pl.counters[8 + d] = x_base;
            pl.counters[10 + d] = 0;
            pl.counters[12 + d] = 0;
        }
    }
    if (tid == 0) {
        pl.counters[0] = n;
        pl.counters[1] = 0;
        pl.counters[2] = 0;
        pl.counters[3] = 0;
    }
}

// ---- the state scans ----------------------------------------------------------------------

constexpr int kScanThreads = 320;
constexpr uint32_t kSOffX = 0;              // x (k or q) -> X_lo
constexpr uint32_t kSOffG = kTile;          // g -> X_hi
constexpr uint32_t kSOffY = 2 * kTile;      // y (v or dO), exact
constexpr uint32_t kSStage = 3 * kTile;
constexpr uint32_t kSOffMisc = 2 * kSStage;
// misc: barriers at 0, the TMEM base at 96, per stage s at 128 + 1024 s: the chunk's
// descriptor (32 B), beta (float[64]) at +64 and P (float[128]) at +320
constexpr uint32_t kSMiscStage = 128;
constexpr uint32_t kScanSmem = kSOffMisc + kSMiscStage + 2 * 1024 + 1024;
static_assert(2 * kScanSmem <= 232448, "two scan CTAs per SM");

// chunk flags: kFirst the piece starts from zero here; kSeed it starts from its slot's state
// here (which is exported as this chunk's state); kPre the state entering the chunk is
// exported; kLast the piece's last chunk; kPost the state after it is exported (the export
// pass: the chain's next chunk's state; the end-state pass: the piece's end state and decay
// product, to its slot); kEnd no more work
enum : int { kFirst = 1, kLast = 2, kPre = 4, kPost = 8, kEnd = 16, kSeed = 32 };

struct SDesc {
    int c, h, flags, lo, hi, slot_pre, slot_post, slot_in;
};

struct ScanParams {
    const __nv_bfloat16* beta;
    float scale;
    int64_t N;
    int32_t H;
    int64_t n_chunks;
    void* ws;
    uint32_t* status;
    int32_t phase;               // 0: the export pass; 1: the end-state pass
};

// kRev = false: x = k, y = v, exports S_in; kRev = true: x = q, y = dO, exports D_end.
template <bool kRev>
__global__ void __launch_bounds__(kScanThreads, 2)
scan_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_g,
            const __grid_constant__ CUtensorMap map_y, const __grid_constant__ ScanParams prm) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* misc = sm + kSOffMisc;
    uint64_t* bars = reinterpret_cast<uint64_t*>(misc);
    uint64_t* bFull = bars + 0;     // [2] TMA bytes + the descriptor
    uint64_t* bProl = bars + 2;     // [2] X ready (4 prologue warps)
    uint64_t* bEmpty = bars + 4;    // [2] the stage's MMAs done
    uint64_t* bReady = bars + 6;    // the state is decayed (4 state warps)
    uint64_t* bSdone = bars + 7;    // the chunk's MMAs done
    uint64_t* bPSync = bars + 8;    // barrier among the prologue warps
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + 96);
    auto stage_misc = [&](uint32_t s) { return misc + kSMiscStage + s * 1024; };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = prm.H;
    const int64_t n_chunks = prm.n_chunks;
    BPlan pl = bplan_view(prm.ws, n_chunks, H);

    if (threadIdx.x == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bFull[s], 2);
            mbar_init(&bProl[s], 4);
            mbar_init(&bEmpty[s], 1);
        }
        mbar_init(bReady, 4);
        mbar_init(bSdone, 1);
        mbar_init(bPSync, 4);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 256);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&map_x);
        tma_prefetch_desc(&map_g);
        tma_prefetch_desc(&map_y);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool timed_out = false;

    if (warp == 0) {
        // ================= producer =================
        const int dn = kRev ? 1 : 0;
        const BDir& bd = pl.dir[dn];
        const bool ends = prm.phase == 1;
        const int n_items = pl.counters[(ends ? 6 : 4) + dn] * H;
        uint32_t it = 0;
        for (;;) {
            int item = 0;
            if (lane == 0) item = atomicAdd(&pl.counters[(ends ? 10 : 1) + dn], 1);
            item = __shfl_sync(0xffffffffu, item, 0);
            const bool done = item >= n_items;
            int c_from = 0, cnt = 1, step = 1, h = 0;
            int2 ch = make_int2(0, 0);
            int4 pc = make_int4(0, 0, 1, -1);
            bool post = false;
            if (!done) {
                pc = bd.pieces[ends ? bd.pieces_a[item / H] : bd.order[item / H]];
                ch = pl.chains[pc.x];
                h = item % H;
                // a chain that is not cut is one piece of any length; cut chains run in pieces
                // of kPiece chunks
                if (!kRev) {
                    c_from = ch.x + pc.y * kPiece;
                    cnt = pc.z == 1 ? ch.y - c_from : min(kPiece, ch.y - c_from);
                    post = ch.y < n_chunks && pl.first_cut[ch.y] > 0;
                } else {
                    const bool head = ch.y < n_chunks && pl.first_cut[ch.y] > 0;
                    c_from = (head ? ch.y : ch.y - 1) - pc.y * kPiece;
                    cnt = c_from - ch.x;               // chunks c_from down to ch.x + 1
                    if (pc.z > 1) cnt = min(kPiece, cnt);
                    step = -1;
                    post = true;
                }
                if (cnt <= 0) continue;
            }
            const bool seeded = !ends && pc.y > 0;     // starts from its slot's state
            const bool last_piece = pc.y == pc.z - 1;
            for (int k = 0; k < cnt; ++k, ++it) {
                const uint32_t s = it & 1;
                const int c = c_from + step * k;
                ChunkMeta meta = {0ull, 0ull};
                __nv_bfloat16 braw[2] = {__float2bfloat16(0.f), __float2bfloat16(0.f)};
                int fc = C;
                if (!done) {
                    meta = pl.meta[c];
                    fc = pl.first_cut[c];
                    if (!kRev) {
#pragma unroll
                        for (int r2 = 0; r2 < 2; ++r2) {
                            const int64_t p = int64_t(c) * C + lane + 32 * r2;
                            if (p < prm.N) braw[r2] = prm.beta[p * H + h];
                        }
                    }
                }
                if (!warp_wait(&bEmpty[s], ((it >> 1) & 1) ^ 1)) { timed_out = true; break; }
                uint8_t* smc = stage_misc(s);
                SDesc* d = reinterpret_cast<SDesc*>(smc);
                uint64_t* bar = &bFull[s];
                if (done) {
                    if (lane == 0) {
                        d->flags = kEnd;
                        mbar_arrive(bar);
                    }
                } else {
                    uint8_t* st = sm + s * kSStage;
                    const int32_t y = int32_t(int64_t(c) * C);
                    if (lane == 0) {
                        mbar_arrive_expect_tx(bar, 3 * kTile);
#pragma unroll
                        for (int p = 0; p < 2; ++p) {
                            tma_load_2d(st + kSOffX + p * kPanel, &map_x, bar, h * D + p * 64, y);
                            tma_load_2d(st + kSOffG + p * kPanel, &map_g, bar, h * D + p * 64, y);
                            tma_load_2d(st + kSOffY + p * kPanel, &map_y, bar, h * D + p * 64, y);
                        }
                    }
                    if (!kRev) {
                        float* beta = reinterpret_cast<float*>(smc + 64);
#pragma unroll
                        for (int r2 = 0; r2 < 2; ++r2) {
                            const int r = lane + 32 * r2;
                            beta[r] = ((meta.valid >> r) & 1ull) ? __bfloat162float(braw[r2]) : 0.f;
                        }
                    }
                    if (lane == 0) {
                        SDesc f;
                        f.c = c;
                        f.h = h;
                        if (k == 0) f.flags = seeded ? (kSeed | kPre) : kFirst;
                        else f.flags = ends ? 0 : kPre;
                        if (k == cnt - 1)
                            f.flags |= kLast | ((ends || (last_piece && post)) ? kPost : 0);
                        if (!kRev) {
                            // the chain's first chunk: only the rows of the segment that reaches
                            // its end (from its last start; none when its last row is padding)
                            const int ls = meta.start ? 63 - __clzll((long long)meta.start) : 0;
                            f.lo = (c == ch.x) ? (((meta.valid >> 63) & 1ull) ? ls : C) : 0;
                            f.hi = C;
                        } else {
                            // the chunk that ends the chain: the rows before its first cut
                            f.lo = 0;
                            f.hi = (c == ch.y) ? fc : C;
                        }
                        f.slot_pre = c;
                        f.slot_post = ends ? pc.w + pc.y : (kRev ? ch.x : ch.y);
                        f.slot_in = pc.w + pc.y - 1;
                        *d = f;
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(bar);
                __syncwarp();
                if (done) break;
            }
            if (done || timed_out) break;
        }
        if (timed_out) set_status(prm.status, KDA_DEV_TIMEOUT);
    } else if (warp == 1) {
        // ================= MMA issuer =================
        const uint32_t sm_addr = smem_u32(sm);
        for (uint32_t it = 0;; ++it) {
            const uint32_t s = it & 1, ph = (it >> 1) & 1;
            if (!warp_wait(&bFull[s], ph)) { timed_out = true; break; }
            const SDesc f = *reinterpret_cast<const SDesc*>(stage_misc(s));
            if (f.flags & kEnd) break;
            if (!warp_wait(&bProl[s], ph)) { timed_out = true; break; }
            if (!warp_wait(bReady, it & 1)) { timed_out = true; break; }
            tc_fence_after();
            const uint32_t st_addr = sm_addr + s * kSStage;
            // S^T (+)= Y^T X: A = Y^T (MN-major), B = X (MN-major), 16 token rows per step
            const uint64_t dY = sdesc_sw128(st_addr + kSOffY, kPanel, 1024);
            const uint64_t dXh = sdesc_sw128(st_addr + kSOffG, kPanel, 1024);
            const uint64_t dXl = sdesc_sw128(st_addr + kSOffX, kPanel, 1024);
            const uint32_t id = idesc_bf16_f32(128, 128, 1, 1);
            const uint32_t acc0 = (f.flags & kFirst) ? 0u : 1u;
            const uint32_t tS = tmem + (it & 1) * 128;      // this chunk's state buffer
#pragma unroll
            for (int kk = 0; kk < C / 16; ++kk)
                mma_bf16(tS, dY + uint64_t(kk * 128), dXh + uint64_t(kk * 128), id, kk > 0 ? 1u : acc0);
#pragma unroll
            for (int kk = 0; kk < C / 16; ++kk)
                mma_bf16(tS, dY + uint64_t(kk * 128), dXl + uint64_t(kk * 128), id, 1u);
            mma_commit(bSdone);
            mma_commit(&bEmpty[s]);
        }
        __syncwarp();
    } else if (warp < 6) {
        // ================= prologue: X = x exp(...) as hi/lo, P =================
        // By channel pairs (2 pm, 2 pm + 1), one thread per pair and half of the rows; the half
        // that the running sum reaches second starts from the other half's sum of g, read
        // before either half overwrites g with X_hi.
        const int pw = threadIdx.x - 64;
        const int lower = pw >> 6;                  // 0: rows 32..63, 1: rows 0..31
        const int c0 = 2 * (pw & 63);
        const float2 l2e = make_float2(kLog2e, kLog2e);
        uint32_t psync_uses = 0;
        for (uint32_t it = 0;; ++it) {
            const uint32_t s = it & 1, ph = (it >> 1) & 1;
            if (!warp_wait(&bFull[s], ph)) { timed_out = true; break; }
            uint8_t* smc = stage_misc(s);
            const SDesc f = *reinterpret_cast<const SDesc*>(smc);
            if (f.flags & kEnd) break;
            uint8_t* st = sm + s * kSStage;
            float* P = reinterpret_cast<float*>(smc + 320);
            // forward: X_t = beta_t k_t exp(Suf_t) on rows t >= lo, walking down from row 63;
            // reverse: X_t = scale q_t exp(G_t) on rows t < hi, walking up from row 0
            float2 run = make_float2(0.f, 0.f);
            const bool second = kRev ? !lower : lower;   // starts from the other half's sum
            if (second) {
                float2 a = make_float2(0.f, 0.f), b = make_float2(0.f, 0.f);
                const int r0 = kRev ? 0 : 32;
#pragma unroll 4
                for (int t = r0; t < r0 + 32; t += 2) {
                    const bool in0 = kRev ? t < f.hi : t >= f.lo;
                    const bool in1 = kRev ? t + 1 < f.hi : t + 1 >= f.lo;
                    if (in0) a = add2(a, unpk2(ld32(st + kSOffG, eoff(t, c0))));
                    if (in1) b = add2(b, unpk2(ld32(st + kSOffG, eoff(t + 1, c0))));
                }
                run = mul2(add2(a, b), l2e);
            }
            if (!group_sync(bPSync, psync_uses, lane)) { timed_out = true; break; }
            if (!kRev) {
                const float* beta = reinterpret_cast<const float*>(smc + 64);
                const int t_hi = lower ? 31 : 63;
#pragma unroll 4
                for (int t = t_hi; t > t_hi - 32; --t) {
                    const uint32_t o = eoff(t, c0);
                    uint32_t hi = 0, lo = 0;
                    if (t >= f.lo) {
                        const float2 x2 = unpk2(ld32(st + kSOffX, o)), g2 = unpk2(ld32(st + kSOffG, o));
                        const float2 e = make_float2(ex2a(run.x), ex2a(run.y));
                        const float2 xv = mul2(mul2(x2, make_float2(beta[t], beta[t])), e);
                        split2(xv.x, xv.y, hi, lo);
                        run = fma2(g2, l2e, run);
                    }
                    st32(st + kSOffG, o, hi);
                    st32(st + kSOffX, o, lo);
                }
            } else {
                const float2 sc2 = make_float2(prm.scale, prm.scale);
                const int t_lo = lower ? 0 : 32;
#pragma unroll 4
                for (int t = t_lo; t < t_lo + 32; ++t) {
                    const uint32_t o = eoff(t, c0);
                    uint32_t hi = 0, lo = 0;
                    if (t < f.hi) {
                        const float2 x2 = unpk2(ld32(st + kSOffX, o)), g2 = unpk2(ld32(st + kSOffG, o));
                        run = fma2(g2, l2e, run);
                        const float2 e = make_float2(ex2a(run.x), ex2a(run.y));
                        const float2 xv = mul2(mul2(x2, sc2), e);
                        split2(xv.x, xv.y, hi, lo);
                    }
                    st32(st + kSOffG, o, hi);
                    st32(st + kSOffX, o, lo);
                }
            }
            if (second) {                               // the chunk's whole decay (used when
                P[c0] = ex2a(run.x);                    // the state goes through the chunk)
                P[c0 + 1] = ex2a(run.y);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bProl[s]);
        }
    } else {
        // ================= state: decay, export =================
        // The state alternates between two TMEM buffers by chunk: the decay step reads the
        // previous chunk's buffer and writes this chunk's, which the MMAs then accumulate
        // into; the export reads the previous buffer after that, while the MMAs run.
        const int qd = warp & 3;                    // TMEM lane quarter
        const int v = qd * 32 + lane;               // value channel (TMEM lane)
        const uint32_t tl = tmem + (uint32_t(qd * 32) << 16);
        uint8_t* const base = reinterpret_cast<uint8_t*>(kRev ? pl.d_end : pl.s_in);
        // The state as the gradient kernel's operand: hi and lo bf16 tiles, 128 x 128 K-major
        // 128B-swizzled (row = key channel), element (key, v) at eoff128(key, v). Lanes v, v + 1
        // swap one value per pair of keys, so that each writes a channel pair of one key (32-bit).
        const int odd = lane & 1;
        const int vv = v - odd;                     // the pair's even value channel
        const uint32_t vbase = uint32_t(vv >> 6) * kPanel128 + uint32_t(vv & 7) * 2;
        const int vg = (vv >> 3) & 7;
        auto export_block = [&](const uint32_t (&r)[32], int cb, uint8_t* dst) {
#pragma unroll
            for (int jp = 0; jp < 16; ++jp) {
                const float x0 = __uint_as_float(r[2 * jp]), x1 = __uint_as_float(r[2 * jp + 1]);
                const float recv = __shfl_xor_sync(0xffffffffu, odd ? x0 : x1, 1);
                const int key = cb * 32 + 2 * jp + odd;
                const uint32_t off = vbase + uint32_t(key) * 128 + (uint32_t(vg ^ (key & 7)) << 4);
                uint32_t hi, lo;
                split2(odd ? recv : x0, odd ? x1 : recv, hi, lo);
                st32(dst, off, hi);
                st32(dst + kTile128, off, lo);
            }
        };
        auto export_state = [&](uint32_t src, uint8_t* dst) {
#pragma unroll 1
            for (int cb = 0; cb < 4; ++cb) {
                uint32_t r[32];
                tmem_ld32(src + cb * 32, r);
                tmem_ld_wait();
                export_block(r, cb, dst);
            }
        };
        // a piece's slot: its state in fp32 (element (key, v) at key * 128 + v) and, after
        // it, the product of its chunks' decays per key channel
        const int dn = kRev ? 1 : 0;
        auto slot_at = [&](int slot, int h) -> float* {
            return reinterpret_cast<float*>(pl.dir[dn].slots + (size_t(slot) * H + h) * kSlotBytes);
        };
        const bool ends = prm.phase == 1;
        float pi = 1.f;                             // (end-state pass) decay product, key v
        uint32_t nd = 0;                            // MMA completions waited for
        for (uint32_t it = 0;; ++it) {
            const uint32_t s = it & 1, ph = (it >> 1) & 1;
            if (!warp_wait(&bFull[s], ph)) { timed_out = true; break; }
            uint8_t* smc = stage_misc(s);
            const SDesc f = *reinterpret_cast<const SDesc*>(smc);
            if (f.flags & kEnd) break;
            const uint32_t cur = tl + (it & 1) * 128, prv = tl + ((it + 1) & 1) * 128;
            const float* P = reinterpret_cast<const float*>(smc + 320);
            if (f.flags & kFirst) {
                pi = 1.f;
                if (ends) {                         // the decay product needs every chunk's P
                    if (!warp_wait(&bProl[s], ph)) { timed_out = true; break; }
                    pi *= P[v];
                }
            } else if (f.flags & kSeed) {
                // the piece's true start state, from its slot: exported as this chunk's entering
                // state, then decayed into this chunk's buffer
                if (!warp_wait(&bProl[s], ph)) { timed_out = true; break; }
                const float* src = slot_at(f.slot_in, f.h) + v;
                uint8_t* dst = base + (size_t(f.slot_pre) * H + f.h) * kStateBytes;
#pragma unroll 1
                for (int cb = 0; cb < 4; ++cb) {
                    uint32_t r[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__ldcg(src + (cb * 32 + j) * D));
                    export_block(r, cb, dst);
#pragma unroll
                    for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * P[cb * 32 + j]);
                    tmem_st32(cur + cb * 32, r);
                }
                tmem_st_wait();
            } else {
                if (!warp_wait(bSdone, nd & 1)) { timed_out = true; break; }
                ++nd;
                if (!warp_wait(&bProl[s], ph)) { timed_out = true; break; }
                tc_fence_after();
                if (ends) pi *= P[v];
#pragma unroll 1
                for (int cb = 0; cb < 4; ++cb) {
                    uint32_t r[32];
                    tmem_ld32(prv + cb * 32, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * P[cb * 32 + j]);
                    tmem_st32(cur + cb * 32, r);
                }
                tmem_st_wait();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bReady);
            if ((f.flags & kPre) && !(f.flags & kSeed))   // the state entering this chunk
                export_state(prv, base + (size_t(f.slot_pre) * H + f.h) * kStateBytes);
            if (f.flags & kLast) {
                if (!warp_wait(bSdone, nd & 1)) { timed_out = true; break; }
                ++nd;
                tc_fence_after();
                if ((f.flags & kPost) && !ends)     // the state after the chain's last chunk
                    export_state(cur, base + (size_t(f.slot_post) * H + f.h) * kStateBytes);
                if ((f.flags & kPost) && ends) {    // the piece's end state and decay product
                    float* dst = slot_at(f.slot_post, f.h);
#pragma unroll 1
                    for (int cb = 0; cb < 4; ++cb) {
                        uint32_t r[32];
                        tmem_ld32(cur + cb * 32, r);
                        tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 32; ++j) __stcg(dst + (cb * 32 + j) * D + v, __uint_as_float(r[j]));
                    }
                    dst[D * D + v] = pi;
                }
            }
            tc_fence_before();
        }
    }
    if (timed_out && lane == 0) set_status(prm.status, KDA_DEV_TIMEOUT);
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 256);
    }
}


// The combine pass between the scans' two passes: per chain cut into pieces and head, the true
// state entering piece j + 1 is T_{j+1} = diag(Pi_j) T_j + E_j (E_j, Pi_j: piece j's end state
// from a zero start and its decay product; T_0 = 0), written over E_j's slot. Each (chain,
// head) spreads over kCombineParts CTAs of 256 threads, 8 state elements per thread (element
// e = key * 128 + v, so key = e >> 7); a step's loads are issued before the previous step's
// stores, so that the steps' memory round trips overlap.
constexpr int kCombineParts = 8;

__global__ void __launch_bounds__(256)
combine_kernel(int64_t n_chunks, int32_t H, int32_t dn, void* ws) {
    BPlan pl = bplan_view(ws, n_chunks, H);
    const BDir& bd = pl.dir[dn];
    const int n = pl.counters[8 + dn] * H * kCombineParts;
    const int tid = threadIdx.x;
    for (int item = blockIdx.x; item < n; item += gridDim.x) {
        const int part = item % kCombineParts;
        const int ih = item / kCombineParts;
        const int4 sp = bd.split[ih / H];
        const int h = ih % H;
        auto slot = [&](int j) {
            return reinterpret_cast<float*>(bd.slots + (size_t(sp.z + j) * H + h) * kSlotBytes);
        };
        int e[8];
#pragma unroll
        for (int m = 0; m < 8; ++m) e[m] = part * 2048 + tid + 256 * m;
        float t[8], ev[8], pv[8];
        const float* e0 = slot(0);                 // T_1 = E_0
#pragma unroll
        for (int m = 0; m < 8; ++m) t[m] = __ldcg(e0 + e[m]);
        if (sp.y > 2) {
            const float* s1 = slot(1);
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                ev[m] = __ldcg(s1 + e[m]);
                pv[m] = __ldcg(s1 + D * D + (e[m] >> 7));
            }
        }
        for (int j = 1; j < sp.y - 1; ++j) {
            float en[8], pn[8];
            if (j + 1 < sp.y - 1) {                // the next step's operands, in flight now
                const float* sn = slot(j + 1);
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    en[m] = __ldcg(sn + e[m]);
                    pn[m] = __ldcg(sn + D * D + (e[m] >> 7));
                }
            }
            float* sj = slot(j);
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                t[m] = fmaf(pv[m], t[m], ev[m]);
                __stcg(sj + e[m], t[m]);
                ev[m] = en[m];
                pv[m] = pn[m];
            }
        }
    }
}

// ---- the gradient kernel ----------------------------------------------------------------

constexpr int kGradThreads = 320;
constexpr uint32_t kGK = 0;                   // k (exact), then with g: S_in_lo
constexpr uint32_t kGG = 1 * kTile;           // g (exact)
constexpr uint32_t kGQL = 2 * kTile;          // q -> Qt_lo
constexpr uint32_t kGQH = 3 * kTile;          // Qt_hi
constexpr uint32_t kGKH = 4 * kTile;          // Ktb_hi
constexpr uint32_t kGKL = 5 * kTile;          // Ktb_lo
constexpr uint32_t kGV = 6 * kTile;           // v (exact)
constexpr uint32_t kGDO = 7 * kTile;          // dO (exact)
constexpr uint32_t kGAH = 8 * kTile;          // A'_hi, 64 x 64 (8 KB); before it, with A'_lo,
constexpr uint32_t kGAL = kGAH + C * C * 2;   //   W_hi and W_lo: D_end_lo
constexpr uint32_t kGWH = kGAL + C * C * 2;   // W_hi
constexpr uint32_t kGWL = kGWH + C * C * 2;   // W_lo
constexpr uint32_t kGSH = kGWL + C * C * 2;   // S_in_hi, 128 x 128 (32 KB)
constexpr uint32_t kGDH = kGSH + kTile128;    // D_end_hi
constexpr uint32_t kGSL = kGK;                // S_in_lo (over k and g)
constexpr uint32_t kGDL = kGAH;               // D_end_lo (over A' and W)
constexpr uint32_t kGMisc = kGDH + kTile128;
// misc: barriers at 0, the TMEM base at 96, beta (float[64], the prologue's) at 128, the
// chunk's base-2 log-decay per key channel (float[128], among the prologue warps) at 384, dg's
// part past the chunk (float[128]) at 896, the epilogue warps'
// dbeta partial sums (float[2][4][8], by block parity) at 1408
constexpr uint32_t kGMiscBytes = 1664;
constexpr uint32_t kGradSmem = kGMisc + kGMiscBytes + 1024;
static_assert(kGradSmem <= 232448, "shared memory per CTA");

// tensor memory (columns)
constexpr uint32_t kTmSC = 0;      // SC, M=64 layout (row t in lane 32 (t/16) + t%16)
constexpr uint32_t kTmW = 64;      // W, M=64 layout
// per buffer b (an item's parity), 192 columns from 128 + 192 b (lane = channel, column = token):
constexpr uint32_t kTmQQ = 128;    //   QQ: Qs^T, then dQ^T's sum (key channel)
constexpr uint32_t kTmKK = 192;    //   KK: T2^T, then dK^T's sum (key channel)
constexpr uint32_t kTmVV = 256;    //   VV: Vs^T, then dV^T's sum (value channel)
constexpr uint32_t kTmBuf = 192;

struct GradParams {
    const __nv_bfloat16* q;          // read again by the epilogue (from L2)
    const __nv_bfloat16* k;
    const __nv_bfloat16* g;
    const __nv_bfloat16* beta;
    float scale;
    int64_t N;
    int32_t H;
    int64_t n_chunks;
    void* ws;
    void* dq;
    void* dk;
    void* dv;
    void* dg;
    void* dbeta;
    uint32_t* status;
};

template <typename To>
__device__ __forceinline__ void store_out(void* base, size_t idx, float x) {
    static_cast<To*>(base)[idx] = from_f32<To>(x);
}

// Bulk copy (no tensor map) of `bytes` (a multiple of 16) from global to shared memory,
// completion signalled on `bar` as transaction bytes.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes),
          "r"(smem_u32(bar))
        : "memory");
}

// mask(SC or W) x mult as hi/lo bf16 tiles (K-major, 64 x 64), by one warp on its TMEM lane
// quarter (rows 16 qd .. 16 qd + 15 of the M=64 accumulator): 16x256b loads give each thread
// rows i0 = 16 qd + lane/4 and i0 + 8 at column pairs 8 r + 2 (lane % 4); stmatrix writes the
// 8x8 blocks.
__device__ __forceinline__ void mask_tiles(uint32_t taddr, uint8_t* t_hi, uint8_t* t_lo,
                                           unsigned long long start, unsigned long long valid,
                                           float mult, int qd, int lane) {
    uint32_t r[32];
    tmem_ld16x256b_x8(taddr, r);
    tmem_ld_wait();
    const int i0 = qd * 16 + (lane >> 2);
    const int sh = 2 * (lane & 3);
    const unsigned long long k0 = keep_bits(start, valid, i0) >> sh;
    const unsigned long long k1 = keep_bits(start, valid, i0 + 8) >> sh;
    uint32_t h0[8], l0[8], h1[8], l1[8];
#pragma unroll
    for (int rp = 0; rp < 8; ++rp) {
        const float a0 = ((k0 >> (8 * rp)) & 1ull) ? mult * __uint_as_float(r[4 * rp]) : 0.f;
        const float b0 = ((k0 >> (8 * rp + 1)) & 1ull) ? mult * __uint_as_float(r[4 * rp + 1]) : 0.f;
        const float a1 = ((k1 >> (8 * rp)) & 1ull) ? mult * __uint_as_float(r[4 * rp + 2]) : 0.f;
        const float b1 = ((k1 >> (8 * rp + 1)) & 1ull) ? mult * __uint_as_float(r[4 * rp + 3]) : 0.f;
        split2(a0, b0, h0[rp], l0[rp]);
        split2(a1, b1, h1[rp], l1[rp]);
    }
    const int mrow = qd * 16 + ((lane >> 3) & 1) * 8 + (lane & 7);
    const uint32_t a_hi = smem_u32(t_hi), a_lo = smem_u32(t_lo);
#pragma unroll
    for (int rp = 0; rp < 8; rp += 2) {
        const int jc = rp + (lane >> 4);
        const uint32_t off = (mrow >> 3) * 1024 + (mrow & 7) * 128 + ((jc ^ (mrow & 7)) << 4);
        stmatrix_x4(a_hi + off, h0[rp], h1[rp], h0[rp + 1], h1[rp + 1]);
        stmatrix_x4(a_lo + off, l0[rp], l1[rp], l0[rp + 1], l1[rp + 1]);
    }
}

// Sum over a warp's 32 lanes of each of v[0..7]: a butterfly that halves the vector at each
// exchange (9 shuffles). Lane l ends up with the sum for entry ((l >> 2) & 7) in lanes with
// (l & 3) == 0.
__device__ __forceinline__ float warp_sum8(float (&v)[8], int lane) {
    float a[4];
    {
        const bool up = lane & 16;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float send = up ? v[e] : v[e + 4];
            const float recv = __shfl_xor_sync(0xffffffffu, send, 16);
            a[e] = (up ? v[e + 4] : v[e]) + recv;
        }
    }
    float b[2];
    {
        const bool up = lane & 8;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const float send = up ? a[e] : a[e + 2];
            const float recv = __shfl_xor_sync(0xffffffffu, send, 8);
            b[e] = (up ? a[e + 2] : a[e]) + recv;
        }
    }
    float x;
    {
        const bool up = lane & 4;
        const float send = up ? b[0] : b[1];
        const float recv = __shfl_xor_sync(0xffffffffu, send, 4);
        x = (up ? b[1] : b[0]) + recv;
    }
    x += __shfl_xor_sync(0xffffffffu, x, 2);
    x += __shfl_xor_sync(0xffffffffu, x, 1);
    return x;
}
// entry of v that warp_sum8 leaves in lane l: bit 16 of l picks the upper half, bit 8 the
// upper quarter, bit 4 the upper eighth
__device__ __forceinline__ int warp_sum8_entry(int lane) {
    return ((lane >> 4) & 1) * 4 + ((lane >> 3) & 1) * 2 + ((lane >> 2) & 1);
}

template <typename To>
__global__ void __launch_bounds__(kGradThreads, 1)
grad_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
            const __grid_constant__ CUtensorMap map_g, const __grid_constant__ CUtensorMap map_v,
            const __grid_constant__ CUtensorMap map_do, const __grid_constant__ GradParams prm) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* misc = sm + kGMisc;
    uint64_t* bars = reinterpret_cast<uint64_t*>(misc);
    uint64_t* bFull = bars + 0;      // q, k, g, v, dO bytes + beta
    uint64_t* bProl = bars + 1;      // Qt, Ktb, P (4 prologue warps)
    uint64_t* bSt = bars + 2;        // S_in and D_end tiles' bytes
    uint64_t* bScores = bars + 3;    // SC and W in TMEM
    uint64_t* bStates = bars + 4;    // the products reading S_in and D_end done
    uint64_t* bMasked = bars + 5;    // A' and W tiles, dg's part past the chunk (4 warps)
    uint64_t* bDone = bars + 6;      // all products done: every tile is free
    uint64_t* bTmemFree = bars + 7;  // [2] the epilogue has read the buffer (4 warps)
    uint64_t* bMiscFree = bars + 9;  // the epilogue has read the carry (4 warps)
    uint64_t* bPSync = bars + 10;    // barrier among the prologue warps
    uint64_t* bESync = bars + 11;    // barrier among the epilogue warps
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + 96);
    float* s_beta = reinterpret_cast<float*>(misc + 128);
    float* s_P = reinterpret_cast<float*>(misc + 384);
    float* s_carry = reinterpret_cast<float*>(misc + 896);
    float* s_dbw = reinterpret_cast<float*>(misc + 1408);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = prm.H;
    const int64_t n_chunks = prm.n_chunks;
    const int64_t n_items = n_chunks * H;
    BPlan pl = bplan_view(prm.ws, n_chunks, H);

    if (threadIdx.x == 0) {
        mbar_init(bFull, 2);
        mbar_init(bProl, 4);
        mbar_init(bSt, 1);
        mbar_init(bScores, 1);
        mbar_init(bStates, 1);
        mbar_init(bMasked, 4);
        mbar_init(bDone, 1);
        mbar_init(&bTmemFree[0], 4);
        mbar_init(&bTmemFree[1], 4);
        mbar_init(bMiscFree, 4);
        mbar_init(bPSync, 4);
        mbar_init(bESync, 4);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&map_q);
        tma_prefetch_desc(&map_k);
        tma_prefetch_desc(&map_g);
        tma_prefetch_desc(&map_v);
        tma_prefetch_desc(&map_do);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool timed_out = false;

    if (warp == 0) {
        // ================= producer =================
        uint32_t n = 0;
        for (int64_t item = blockIdx.x; item < n_items; item += gridDim.x, ++n) {
            const int c = int(item / H), h = int(item % H);
            const unsigned long long valid = pl.meta[c].valid;
            const bool cin = pl.first_cut[c] > 0;
            const bool cout = (c + 1 < n_chunks) && pl.first_cut[c + 1] > 0;
            __nv_bfloat16 braw[2] = {__float2bfloat16(0.f), __float2bfloat16(0.f)};
#pragma unroll
            for (int r2 = 0; r2 < 2; ++r2) {
                const int64_t p = int64_t(c) * C + lane + 32 * r2;
                if (p < prm.N) braw[r2] = prm.beta[p * H + h];
            }
            // every tile is free once the previous item's products are done (the epilogue
            // reads only tensor memory and L2)
            if (n > 0 && !warp_wait(bDone, (n - 1) & 1)) { timed_out = true; break; }
            const int32_t y = int32_t(int64_t(c) * C);
            const uint8_t* st_s = reinterpret_cast<const uint8_t*>(pl.s_in) + (size_t(c) * H + h) * kStateBytes;
            const uint8_t* st_d = reinterpret_cast<const uint8_t*>(pl.d_end) + (size_t(c) * H + h) * kStateBytes;
            if (lane == 0) {
                mbar_arrive_expect_tx(bFull, 5 * kTile);
#pragma unroll
                for (int p = 0; p < 2; ++p) {
                    const int32_t x = h * D + p * 64;
                    tma_load_2d(sm + kGK + p * kPanel, &map_k, bFull, x, y);
                    tma_load_2d(sm + kGG + p * kPanel, &map_g, bFull, x, y);
                    tma_load_2d(sm + kGQL + p * kPanel, &map_q, bFull, x, y);
                    tma_load_2d(sm + kGV + p * kPanel, &map_v, bFull, x, y);
                    tma_load_2d(sm + kGDO + p * kPanel, &map_do, bFull, x, y);
                }
                const uint32_t st_bytes = (cin ? 2 * kTile128 : 0u) + (cout ? 2 * kTile128 : 0u);
                if (st_bytes) {
                    mbar_arrive_expect_tx(bSt, st_bytes);
                    if (cout) {
                        bulk_load(sm + kGDH, st_d, kTile128, bSt);
                        bulk_load(sm + kGDL, st_d + kTile128, kTile128, bSt);
                    }
                    if (cin) bulk_load(sm + kGSH, st_s, kTile128, bSt);
                } else {
                    mbar_arrive(bSt);
                }
            }
#pragma unroll
            for (int r2 = 0; r2 < 2; ++r2) {
                const int r = lane + 32 * r2;
                s_beta[r] = ((valid >> r) & 1ull) ? __bfloat162float(braw[r2]) : 0.f;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bFull);
            // S_in_lo goes over k and g once the prologue has read them
            if (!warp_wait(bProl, n & 1)) { timed_out = true; break; }
            if (lane == 0 && cin) bulk_load(sm + kGSL, st_s + kTile128, kTile128, bSt);
            __syncwarp();
        }
        // copies still in flight when a wait gave up: wait for them (bounded) before exiting
        if (timed_out && n > 0) {
            (void)warp_wait(bFull, (n - 1) & 1);
            (void)warp_wait(bSt, (n - 1) & 1);
        }
    } else if (warp == 1) {
        // ================= MMA issuer =================
        const uint32_t a = smem_u32(sm);
        const uint64_t dK_H = sdesc_sw128(a + kGKH, 16, 1024), dK_L = sdesc_sw128(a + kGKL, 16, 1024);
        const uint64_t dQ_H = sdesc_sw128(a + kGQH, 16, 1024), dQ_L = sdesc_sw128(a + kGQL, 16, 1024);
        const uint64_t dDO = sdesc_sw128(a + kGDO, 16, 1024), dV = sdesc_sw128(a + kGV, 16, 1024);
        const uint64_t dSH = sdesc_sw128(a + kGSH, 16, 1024), dSL = sdesc_sw128(a + kGSL, 16, 1024);
        const uint64_t dDH = sdesc_sw128(a + kGDH, 16, 1024), dDL = sdesc_sw128(a + kGDL, 16, 1024);
        const uint64_t mDH = sdesc_sw128(a + kGDH, kPanel128, 1024);      // D_end^T (MN-major)
        const uint64_t mDL = sdesc_sw128(a + kGDL, kPanel128, 1024);
        const uint64_t mK_H = sdesc_sw128(a + kGKH, kPanel, 1024), mK_L = sdesc_sw128(a + kGKL, kPanel, 1024);
        const uint64_t mQ_H = sdesc_sw128(a + kGQH, kPanel, 1024), mQ_L = sdesc_sw128(a + kGQL, kPanel, 1024);
        const uint64_t mDO = sdesc_sw128(a + kGDO, kPanel, 1024);
        const uint64_t dW_H = sdesc_sw128(a + kGWH, 16, 1024), dW_L = sdesc_sw128(a + kGWL, 16, 1024);
        const uint64_t mW_H = sdesc_sw128(a + kGWH, kPanel, 1024), mW_L = sdesc_sw128(a + kGWL, kPanel, 1024);
        const uint64_t mA_H = sdesc_sw128(a + kGAH, kPanel, 1024), mA_L = sdesc_sw128(a + kGAL, kPanel, 1024);
        const uint32_t id64 = idesc_bf16_f32(64, 64, 0, 0);
        const uint32_t idKK = idesc_bf16_f32(128, 64, 0, 0);
        const uint32_t idMK = idesc_bf16_f32(128, 64, 1, 0);
        const uint32_t idMM = idesc_bf16_f32(128, 64, 1, 1);
        uint32_t n = 0;
        for (int64_t item = blockIdx.x; item < n_items; item += gridDim.x, ++n) {
            const int c = int(item / H);
            const bool cin = pl.first_cut[c] > 0;
            const bool cout = (c + 1 < n_chunks) && pl.first_cut[c + 1] > 0;
            const uint32_t ph = n & 1;
            if (!warp_wait(bFull, ph)) { timed_out = true; break; }
            tc_fence_after();
            // W = dO V^T (its TMEM columns are free: the previous item's masking read them
            // before its last products)
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
                mma_bf16(tmem + kTmW, dDO + kofs64(kk), dV + kofs64(kk), id64, kk > 0 ? 1u : 0u);
            if (!warp_wait(bProl, ph)) { timed_out = true; break; }
            tc_fence_after();
            // SC = Qt Ktb^T as hi*hi + hi*lo + lo*hi
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
                mma_bf16(tmem + kTmSC, dQ_H + kofs64(kk), dK_H + kofs64(kk), id64, kk > 0 ? 1u : 0u);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
                mma_bf16(tmem + kTmSC, dQ_H + kofs64(kk), dK_L + kofs64(kk), id64, 1u);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
                mma_bf16(tmem + kTmSC, dQ_L + kofs64(kk), dK_H + kofs64(kk), id64, 1u);
            mma_commit(bScores);
            // the buffer's previous user is the item two back: its epilogue must have read it
            const uint32_t tb = tmem + (n & 1) * kTmBuf;
            if (!warp_wait(bSt, ph)) { timed_out = true; break; }
            if (!warp_wait(&bTmemFree[n & 1], ((n >> 1) & 1) ^ 1)) { timed_out = true; break; }
            tc_fence_after();
            if (cin) {           // QQ = Qs^T = S_in dO^T
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_bf16(tb + kTmQQ, dSH + kofs128(kk), dDO + kofs64(kk), idKK, kk > 0 ? 1u : 0u);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_bf16(tb + kTmQQ, dSL + kofs128(kk), dDO + kofs64(kk), idKK, 1u);
            }
            if (cout) {          // KK = T2^T = D_end V^T;  VV = Vs^T = D_end^T Ktb^T
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_bf16(tb + kTmKK, dDH + kofs128(kk), dV + kofs64(kk), idKK, kk > 0 ? 1u : 0u);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_bf16(tb + kTmKK, dDL + kofs128(kk), dV + kofs64(kk), idKK, 1u);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_bf16(tb + kTmVV, mDH + uint64_t(kk * 128), dK_H + kofs64(kk), idMK, kk > 0 ? 1u : 0u);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_bf16(tb + kTmVV, mDH + uint64_t(kk * 128), dK_L + kofs64(kk), idMK, 1u);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_bf16(tb + kTmVV, mDL + uint64_t(kk * 128), dK_H + kofs64(kk), idMK, 1u);
            }
            mma_commit(bStates);     // D_end_lo's space is the A' and W tiles'
            if (!warp_wait(bMasked, ph)) { timed_out = true; break; }
            tc_fence_after();
            const uint32_t aq = cin ? 1u : 0u, akv = cout ? 1u : 0u;   // onto the state terms
            // QQ += Ktb^T W^T  (K = 64 tokens s; W^T's K-major rows are W's rows)
#pragma unroll
            for (int kk = 0; kk < C / 16; ++kk)
                mma_bf16(tb + kTmQQ, mK_H + uint64_t(kk * 128), dW_H + uint64_t(kk * 2), idMK, kk > 0 ? 1u : aq);
#pragma unroll
            for (int kk = 0; kk < C / 16; ++kk)
                mma_bf16(tb + kTmQQ, mK_H + uint64_t(kk * 128), dW_L + uint64_t(kk * 2), idMK, 1u);
#pragma unroll
            for (int kk = 0; kk < C / 16; ++kk)
                mma_bf16(tb + kTmQQ, mK_L + uint64_t(kk * 128), dW_H + uint64_t(kk * 2), idMK, 1u);
            // KK += Qt^T W  (K = 64 tokens t; Qt carries scale)
#pragma unroll
            for (int kk = 0; kk < C / 16; ++kk)
                mma_bf16(tb + kTmKK, mQ_H + uint64_t(kk * 128), mW_H + uint64_t(kk * 128), idMM, kk > 0 ? 1u : akv);
#pragma unroll
            for (int kk = 0; kk < C / 16; ++kk)
                mma_bf16(tb + kTmKK, mQ_H + uint64_t(kk * 128), mW_L + uint64_t(kk * 128), idMM, 1u);
#pragma unroll
            for (int kk = 0; kk < C / 16; ++kk)
                mma_bf16(tb + kTmKK, mQ_L + uint64_t(kk * 128), mW_H + uint64_t(kk * 128), idMM, 1u);
            // VV += dO^T A'  (K = 64 tokens t)
#pragma unroll
            for (int kk = 0; kk < C / 16; ++kk)
                mma_bf16(tb + kTmVV, mDO + uint64_t(kk * 128), mA_H + uint64_t(kk * 128), idMM, kk > 0 ? 1u : akv);
#pragma unroll
            for (int kk = 0; kk < C / 16; ++kk)
                mma_bf16(tb + kTmVV, mDO + uint64_t(kk * 128), mA_L + uint64_t(kk * 128), idMM, 1u);
            mma_commit(bDone);
        }
        __syncwarp();
    } else if (warp < 6) {
        // ================= prologue: Qt, Ktb (hi/lo), P; the A' and W tiles; the carry =======
        const int qd = warp & 3;                 // TMEM lane quarter
        const int ch = qd * 32 + lane;           // key channel (= TMEM lane of T2)
        const uint32_t tl = tmem + (uint32_t(qd * 32) << 16);
        uint32_t psync_uses = 0;
        uint32_t n = 0;
        for (int64_t item = blockIdx.x; item < n_items; item += gridDim.x, ++n) {
            const int c = int(item / H);
            const ChunkMeta meta = pl.meta[c];
            const int fc = pl.first_cut[c];
            const bool cout = (c + 1 < n_chunks) && pl.first_cut[c + 1] > 0;
            const int lo_last = meta.start ? 63 - __clzll((long long)meta.start) : 0;
            const uint32_t ph = n & 1;
            if (!warp_wait(bFull, ph)) { timed_out = true; break; }
            // Qt and Ktb by channel pairs (2 pm, 2 pm + 1): one thread per pair and half of the
            // rows, the lower half starting from the sum of g over the upper half's real rows
            {
                const int pw = threadIdx.x - 64;
                const int lower = pw >> 6;               // 0: rows 63..32, 1: rows 31..0
                const int c0 = 2 * (pw & 63);
                float2 suf2 = make_float2(0.f, 0.f);
                if (lower) {
                    float2 a = make_float2(0.f, 0.f), b = make_float2(0.f, 0.f);
#pragma unroll 4
                    for (int t = 32; t < C; t += 2) {
                        if ((meta.valid >> t) & 1ull) a = add2(a, unpk2(ld32(sm + kGG, eoff(t, c0))));
                        if ((meta.valid >> (t + 1)) & 1ull) b = add2(b, unpk2(ld32(sm + kGG, eoff(t + 1, c0))));
                    }
                    suf2 = mul2(add2(a, b), make_float2(kLog2e, kLog2e));
                }
                const float2 sc2 = make_float2(prm.scale, prm.scale);
                const float2 l2e = make_float2(kLog2e, kLog2e);
                const int t_hi = lower ? 31 : 63;
#pragma unroll 4
                for (int t = t_hi; t > t_hi - 32; --t) {
                    const uint32_t o = eoff(t, c0);
                    uint32_t qh = 0, ql = 0, kh = 0, kl = 0;
                    if ((meta.valid >> t) & 1ull) {
                        const float2 q2 = unpk2(ld32(sm + kGQL, o)), k2 = unpk2(ld32(sm + kGK, o));
                        const float2 g2 = unpk2(ld32(sm + kGG, o));
                        const float2 eN = make_float2(ex2a(-suf2.x), ex2a(-suf2.y));
                        const float2 eS = make_float2(ex2a(suf2.x), ex2a(suf2.y));
                        const float2 qt = mul2(mul2(q2, sc2), eN);
                        const float2 kt = mul2(mul2(k2, make_float2(s_beta[t], s_beta[t])), eS);
                        split2(qt.x, qt.y, qh, ql);
                        split2(kt.x, kt.y, kh, kl);
                        suf2 = fma2(g2, l2e, suf2);
                    }
                    st32(sm + kGQH, o, qh);
                    st32(sm + kGQL, o, ql);
                    st32(sm + kGKH, o, kh);
                    st32(sm + kGKL, o, kl);
                }
                if (lower) {                             // the chunk's whole real g
                    s_P[c0] = suf2.x;
                    s_P[c0 + 1] = suf2.y;
                }
            }
            if (!group_sync(bPSync, psync_uses, lane)) { timed_out = true; break; }
            const float suf = s_P[ch];
            // (the next item rewrites s_P)
            if (!group_sync(bPSync, psync_uses, lane)) { timed_out = true; break; }
            // a channel whose chunk log-decay is below -80: the factorised products lose it,
            // so the item goes to the fp32 redo, which rewrites its gradients
            const bool out_of_range = __any_sync(0xffffffffu, suf < kRangeLog2);
            if (out_of_range && lane == 0 && atomicExch(&pl.redo_flag[item], 1) == 0)
                pl.redo[atomicAdd(&pl.counters[3], 1)] = int32_t(item);
            const float Pch = ex2a(suf);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bProl);
            // dg's part past the chunk, when its last segment goes on: rowdot(S_out, D_end) =
            // [no cut] P rowdot(S_in, D_end) + sum over the last segment's rows s of Ktb_s T2_s
            float carry = 0.f;
            if (!warp_wait(bSt, ph)) { timed_out = true; break; }
            if (cout && fc == C) {
                float acc4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
                for (int gi = 0; gi < 16; ++gi) {
                    float& acc = acc4[gi & 3];
                    const uint32_t off = eoff128(ch, gi * 8);
                    const uint4 sh = *reinterpret_cast<const uint4*>(sm + kGSH + off);
                    const uint4 sl = *reinterpret_cast<const uint4*>(sm + kGSL + off);
                    const uint4 dh = *reinterpret_cast<const uint4*>(sm + kGDH + off);
                    const uint4 dl = *reinterpret_cast<const uint4*>(sm + kGDL + off);
                    const uint32_t a4[4] = {sh.x, sh.y, sh.z, sh.w}, b4[4] = {sl.x, sl.y, sl.z, sl.w};
                    const uint32_t c4[4] = {dh.x, dh.y, dh.z, dh.w}, d4[4] = {dl.x, dl.y, dl.z, dl.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float s0 = __uint_as_float(a4[e] << 16) + __uint_as_float(b4[e] << 16);
                        const float s1 = __uint_as_float(a4[e] & 0xffff0000u) + __uint_as_float(b4[e] & 0xffff0000u);
                        const float d0 = __uint_as_float(c4[e] << 16) + __uint_as_float(d4[e] << 16);
                        const float d1 = __uint_as_float(c4[e] & 0xffff0000u) + __uint_as_float(d4[e] & 0xffff0000u);
                        acc = fmaf(s0, d0, acc);
                        acc = fmaf(s1, d1, acc);
                    }
                }
                carry = Pch * ((acc4[0] + acc4[1]) + (acc4[2] + acc4[3]));
            }
            if (!warp_wait(bScores, ph)) { timed_out = true; break; }
            if (!warp_wait(bStates, ph)) { timed_out = true; break; }
            tc_fence_after();
            const uint32_t tb = tl + (n & 1) * kTmBuf;
            if (cout) {
                float cacc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
                for (int hb = lo_last >> 5; hb < 2; ++hb) {
                    uint32_t t2[32];
                    tmem_ld32(tb + kTmKK + hb * 32, t2);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int s = hb * 32 + j;
                        if (s >= lo_last) {
                            const uint32_t o = eoff(s, ch);
                            const float kt = ld_bf(sm + kGKH, o) + ld_bf(sm + kGKL, o);
                            cacc[j & 3] = fmaf(kt, __uint_as_float(t2[j]), cacc[j & 3]);
                        }
                    }
                }
                carry += (cacc[0] + cacc[1]) + (cacc[2] + cacc[3]);
            }
            // the state terms, in place, before the products that accumulate onto them: QQ =
            // P Qs^T on the carried rows (t < fc; S_dec = diag(P) S_in), KK and VV on the last
            // segment's rows (t >= lo_last), zero elsewhere
            if (fc > 0) {
#pragma unroll 1
                for (int hb = 0; hb < 2; ++hb) {
                    uint32_t r[32];
                    tmem_ld32(tb + kTmQQ + hb * 32, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        r[j] = (hb * 32 + j < fc) ? __float_as_uint(Pch * __uint_as_float(r[j])) : 0u;
                    tmem_st32(tb + kTmQQ + hb * 32, r);
                }
            }
            if (cout && lo_last > 0) {
                const uint32_t zero[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
#pragma unroll 1
                for (int blk = 0; blk < (lo_last >> 3); ++blk) {
                    tmem_st8(tb + kTmKK + blk * 8, zero);
                    tmem_st8(tb + kTmVV + blk * 8, zero);
                }
                const int b0 = lo_last & ~7;
                if (b0 < lo_last) {
                    uint32_t rk[8], rv[8];
                    tmem_ld8(tb + kTmKK + b0, rk);
                    tmem_ld8(tb + kTmVV + b0, rv);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        if (b0 + j < lo_last) {
                            rk[j] = 0u;
                            rv[j] = 0u;
                        }
                    }
                    tmem_st8(tb + kTmKK + b0, rk);
                    tmem_st8(tb + kTmVV + b0, rv);
                }
            }
            tmem_st_wait();
            // the carry is the previous item's until its epilogue has read it
            if (n > 0 && !warp_wait(bMiscFree, (n - 1) & 1)) { timed_out = true; break; }
            s_carry[ch] = carry;
            // A' = mask(SC) (Qt carries scale), W = mask(W) as hi/lo tiles, over D_end_lo once
            // it is read
            mask_tiles(tl + kTmSC, sm + kGAH, sm + kGAL, meta.start, meta.valid, 1.f, qd, lane);
            mask_tiles(tl + kTmW, sm + kGWH, sm + kGWL, meta.start, meta.valid, 1.f, qd, lane);
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bMasked);
        }
    } else {
        // ================= epilogue: tensor memory and L2 only =================
        const int qd = warp & 3;                 // TMEM lane quarter
        const int wr = warp - 6;
        const int i = qd * 32 + lane;            // key channel (dq, dk, dg) / value channel (dv)
        const uint32_t tl = tmem + (uint32_t(qd * 32) << 16);
        const float scale = prm.scale;
        const size_t row_stride = size_t(H) * D;
        uint32_t esync_uses = 0;
        uint32_t n = 0;
        for (int64_t item = blockIdx.x; item < n_items; item += gridDim.x, ++n) {
            const int c = int(item / H), h = int(item % H);
            const ChunkMeta meta = pl.meta[c];
            const uint32_t ph = n & 1;
            const uint32_t tb = tl + (n & 1) * kTmBuf;
            if (!warp_wait(bMasked, ph)) { timed_out = true; break; }
            if (!warp_wait(bDone, ph)) { timed_out = true; break; }
            tc_fence_after();
            float run = s_carry[i];              // dg's running sum, from the chunk's end
            __syncwarp();
            if (lane == 0) mbar_arrive(bMiscFree);
            const int64_t row0 = int64_t(c) * C;
            const int t_end = int(prm.N - row0 < C ? prm.N - row0 : C);   // tokens that exist
            // this thread's element of token t: base + t * H * 128 (32-bit offsets)
            const size_t ebase = size_t(row0) * row_stride + size_t(h) * D + i;
            const uint32_t tstride = uint32_t(row_stride);
            const __nv_bfloat16* qp = prm.q + ebase;
            const __nv_bfloat16* kp = prm.k + ebase;
            const __nv_bfloat16* gp = prm.g + ebase;
            const __nv_bfloat16* bp = prm.beta + size_t(row0) * H + h;
            float suf = 0.f;
            // k, g, q and beta of the block, one block ahead
            __nv_bfloat16 kn[8], gn[8], qn[8], bn[8];
            auto fetch = [&](int t0) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int t = t0 + j;
                    const __nv_bfloat16 z = __float2bfloat16(0.f);
                    const bool ok = t < t_end;
                    kn[j] = ok ? kp[uint32_t(t) * tstride] : z;
                    gn[j] = ok ? gp[uint32_t(t) * tstride] : z;
                    qn[j] = ok ? qp[uint32_t(t) * tstride] : z;
                    bn[j] = ok ? bp[uint32_t(t) * uint32_t(H)] : z;
                }
            };
            fetch(56);
#pragma unroll 1
            for (int blk = 7; blk >= 0; --blk) {
                __nv_bfloat16 kb[8], gb[8], qb[8];
                float bb[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    kb[j] = kn[j];
                    gb[j] = gn[j];
                    qb[j] = qn[j];
                    bb[j] = ((meta.valid >> (blk * 8 + j)) & 1ull) ? __bfloat162float(bn[j]) : 0.f;
                }
                if (blk > 0) fetch((blk - 1) * 8);
                uint32_t aQ[8], aK[8], aV[8];
                tmem_ld8(tb + kTmQQ + blk * 8, aQ);
                tmem_ld8(tb + kTmKK + blk * 8, aK);
                tmem_ld8(tb + kTmVV + blk * 8, aV);
                tmem_ld_wait();
                float db[8];
#pragma unroll
                for (int j = 7; j >= 0; --j) {
                    const int t = blk * 8 + j;
                    float dq = 0.f, dk = 0.f, dv = 0.f, dg = 0.f;
                    db[j] = 0.f;
                    if ((meta.valid >> t) & 1ull) {
                        // QQ = W Ktb + [carried] P Qs, KK = scale Qt^T W + [last] T2,
                        // VV = A'^T dO + [last] Vs (the masks and P applied in tensor memory)
                        const float qsum = __uint_as_float(aQ[j]);
                        const float ksum = __uint_as_float(aK[j]);
                        const float eS = ex2a(suf), eN = ex2a(-suf);
                        dq = scale * eN * qsum;
                        const float dkr = eS * ksum;
                        const float kv = __bfloat162float(kb[j]);
                        dk = bb[j] * dkr;
                        dv = __uint_as_float(aV[j]);
                        db[j] = kv * dkr;
                        // q dq - k dk = scale Qt qsum - Ktb ksum
                        run += scale * (__bfloat162float(qb[j]) * eN) * qsum - (bb[j] * kv * eS) * ksum;
                        const bool is_start = (meta.start >> t) & 1ull;
                        dg = is_start ? 0.f : run;
                        if (is_start) run = 0.f;
                        suf += __bfloat162float(gb[j]) * kLog2e;
                    } else {
                        run = 0.f;
                    }
                    if (t < t_end) {
                        const size_t idx = ebase + uint32_t(t) * tstride;
                        store_out<To>(prm.dq, idx, dq);
                        store_out<To>(prm.dk, idx, dk);
                        store_out<To>(prm.dv, idx, dv);
                        store_out<To>(prm.dg, idx, dg);
                    }
                }
                // dbeta_t = sum over the 128 key channels: this warp's 32, then the 4 warps'
                // partial sums in a fixed order (the result does not depend on timing)
                const float part = warp_sum8(db, lane);
                float* buf = s_dbw + (blk & 1) * 32;
                if ((lane & 3) == 0) buf[wr * 8 + warp_sum8_entry(lane)] = part;
                if (!group_sync(bESync, esync_uses, lane)) { timed_out = true; break; }
                if (wr == 0 && lane < 8) {
                    const int t = blk * 8 + lane;
                    const float sum = ((buf[lane] + buf[8 + lane]) + buf[16 + lane]) + buf[24 + lane];
                    if (t < t_end) store_out<To>(prm.dbeta, size_t(row0 + t) * H + h, sum);
                }
            }
            if (timed_out) break;
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bTmemFree[n & 1]);
        }
    }
    if (timed_out && lane == 0) set_status(prm.status, KDA_DEV_TIMEOUT);
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}


// ---- the fp32 redo of items outside the factorised form's range -------------------------
// A (chunk, head) item whose chunk log-decay falls below -80 on some key channel is listed
// by the gradient kernel; this kernel rewrites its gradients with the token recurrence of
// the chunk in fp32: forward from S_in (the walks' dq_t = scale S_t do_t), then backward
// from D_end (A_t = scale q_t do_t^T + exp(g_{t+1}) A_{t+1}: dk = beta A v, dv = beta A^T k,
// dbeta = k^T A v, dg the running sum of q dq - k dk plus rowdot(S_out, D_end) on the last
// segment). One CTA of 128 threads per item; the states S and A sit in shared memory with
// rows padded to 129 floats, so that row and column sweeps are both free of bank conflicts.
// It exits at once when nothing is listed.

constexpr int kRedoThreads = 128;
constexpr int kRS = D + 1;
constexpr uint32_t kRedoSmem = uint32_t(2 * D * kRS + C * D + 6 * D + 32) * 4;

struct RedoParams {
    const __nv_bfloat16* q;
    const __nv_bfloat16* k;
    const __nv_bfloat16* v;
    const __nv_bfloat16* g;
    const __nv_bfloat16* beta;
    const __nv_bfloat16* d_o;
    float scale;
    int64_t N;
    int32_t H;
    int64_t n_chunks;
    void* ws;
    void* dq;
    void* dk;
    void* dv;
    void* dg;
    void* dbeta;
};

template <typename To>
__global__ void __launch_bounds__(kRedoThreads)
redo_kernel(const __grid_constant__ RedoParams prm) {
    extern __shared__ float rsm[];
    float* S = rsm;                     // [128][129] the state (row = key channel)
    float* A = S + D * kRS;             // [128][129] the adjoint
    float* dqs = A + D * kRS;           // [64][128] dq of the chunk's rows
    float* vk = dqs + C * D;            // the current token's k, v, q, dO, g
    float* vv = vk + D;
    float* vq = vv + D;
    float* vo = vq + D;
    float* vg = vo + D;
    float* vu = vg + D;                 // (A v) per key channel
    float* red = vu + D;                // [4] dbeta's partial sums
    const int i = threadIdx.x, lane = i & 31, warp = i >> 5;
    const int H = prm.H;
    BPlan pl = bplan_view(prm.ws, prm.n_chunks, H);
    const int n = pl.counters[3];
    const float scale = prm.scale;
    for (int r = blockIdx.x; r < n; r += gridDim.x) {
        const int item = pl.redo[r];
        const int c = item / H, h = item % H;
        const ChunkMeta meta = pl.meta[c];
        const bool cin = pl.first_cut[c] > 0;
        const bool cout = (c + 1 < prm.n_chunks) && pl.first_cut[c + 1] > 0;
        const int64_t row0 = int64_t(c) * C;
        const uint8_t* ts = reinterpret_cast<const uint8_t*>(pl.s_in) + (size_t(c) * H + h) * kStateBytes;
        const uint8_t* td = reinterpret_cast<const uint8_t*>(pl.d_end) + (size_t(c) * H + h) * kStateBytes;
        auto tok = [&](int t) -> size_t { return (size_t(row0 + t) * H + h) * D; };
        for (int j = 0; j < D; ++j) {
            const uint32_t o = eoff128(i, j);
            S[i * kRS + j] = cin ? ld_bf(ts, o) + ld_bf(ts + kTile128, o) : 0.f;
        }
        // forward: S_t and dq_t
        for (int t = 0; t < C; ++t) {
            const bool real = (meta.valid >> t) & 1ull;
            __syncthreads();
            if (real) {
                const size_t b = tok(t) + i;
                vk[i] = __bfloat162float(prm.k[b]);
                vv[i] = __bfloat162float(prm.v[b]);
                vo[i] = __bfloat162float(prm.d_o[b]);
                vg[i] = __bfloat162float(prm.g[b]);
            }
            __syncthreads();
            float dq = 0.f;
            float* Si = S + i * kRS;
            if (real) {
                const bool start = (meta.start >> t) & 1ull;
                const float e = start ? 0.f : expf(vg[i]);
                const float bk = __bfloat162float(prm.beta[size_t(row0 + t) * H + h]) * vk[i];
                float acc = 0.f;
                for (int j = 0; j < D; ++j) {
                    const float sv = fmaf(e, Si[j], bk * vv[j]);
                    Si[j] = sv;
                    acc = fmaf(sv, vo[j], acc);
                }
                dq = scale * acc;
            } else {
                for (int j = 0; j < D; ++j) Si[j] = 0.f;
            }
            dqs[t * D + i] = dq;
        }
        // the adjoint at the chunk's end, and dg's part past the chunk
        float run = 0.f;
        {
            float* Ai = A + i * kRS;
            const float* Si = S + i * kRS;
            for (int j = 0; j < D; ++j) {
                const uint32_t o = eoff128(i, j);
                const float a = cout ? ld_bf(td, o) + ld_bf(td + kTile128, o) : 0.f;
                Ai[j] = a;
                run = fmaf(Si[j], a, run);
            }
        }
        // backward: A_t, dk, dv, dbeta, dg
        for (int t = C - 1; t >= 0; --t) {
            const bool real = (meta.valid >> t) & 1ull;
            const bool start = (meta.start >> t) & 1ull;
            const float bt = real ? __bfloat162float(prm.beta[size_t(row0 + t) * H + h]) : 0.f;
            __syncthreads();
            if (real) {
                const size_t b = tok(t) + i;
                vk[i] = __bfloat162float(prm.k[b]);
                vv[i] = __bfloat162float(prm.v[b]);
                vq[i] = __bfloat162float(prm.q[b]);
                vo[i] = __bfloat162float(prm.d_o[b]);
                vg[i] = __bfloat162float(prm.g[b]);
            }
            __syncthreads();
            float* Ai = A + i * kRS;
            if (real) {
                const float sq = scale * vq[i];
                float u = 0.f;
                for (int j = 0; j < D; ++j) {
                    const float a = fmaf(sq, vo[j], Ai[j]);
                    Ai[j] = a;
                    u = fmaf(a, vv[j], u);
                }
                vu[i] = u;
            }
            __syncthreads();
            float dq = 0.f, dk = 0.f, dv = 0.f, dg = 0.f, dbp = 0.f;
            if (real) {
                for (int kk = 0; kk < D; ++kk) dv = fmaf(A[kk * kRS + i], vk[kk], dv);   // column i
                dv *= bt;
                dq = dqs[t * D + i];
                dk = bt * vu[i];
                dbp = vk[i] * vu[i];
                run += vq[i] * dq - vk[i] * dk;
                dg = start ? 0.f : run;
                if (start) run = 0.f;
            } else {
                run = 0.f;
            }
#pragma unroll
            for (int m = 16; m > 0; m >>= 1) dbp += __shfl_xor_sync(0xffffffffu, dbp, m);
            if (lane == 0) red[warp] = dbp;
            if (row0 + t < prm.N) {
                const size_t b = tok(t) + i;
                store_out<To>(prm.dq, b, dq);
                store_out<To>(prm.dk, b, dk);
                store_out<To>(prm.dv, b, dv);
                store_out<To>(prm.dg, b, dg);
            }
            __syncthreads();
            if (i == 0 && row0 + t < prm.N)
                store_out<To>(prm.dbeta, size_t(row0 + t) * H + h, (red[0] + red[1]) + (red[2] + red[3]));
            // the adjoint handed to row t - 1: exp(g_t) A_t within the segment, else none
            const float e = (real && !start) ? expf(vg[i]) : 0.f;
            for (int j = 0; j < D; ++j) Ai[j] *= e;
        }
        __syncthreads();
    }
}

}  // namespace tcb

size_t bwd_tc_workspace_bytes(int64_t N, int32_t H) {
    const int64_t n_chunks = ceil_div(N, kChunk);
    return tcb::bplan_bytes(n_chunks, H) + 2 * size_t(n_chunks) * H * tcb::kStateBytes;
}

kda_status_t launch_bwd_tc(const void* q, const void* k, const void* v, const void* g,
                           const void* beta, const void* d_o, const int32_t* seg, int64_t B,
                           int64_t T_len, int32_t H, float scale, kda_dtype_t grad_dtype,
                           void* dq, void* dk, void* dv, void* dg, void* dbeta, void* ws,
                           uint32_t* status_dev, cudaStream_t stream) {
    using namespace tcb;
    const int64_t N = B * T_len;
    const int64_t n_chunks = ceil_div(N, C);
    CUtensorMap m[5];
    if (!tc::make_map(&m[0], q, N, H) || !tc::make_map(&m[1], k, N, H) ||
        !tc::make_map(&m[2], g, N, H) || !tc::make_map(&m[3], v, N, H) ||
        !tc::make_map(&m[4], d_o, N, H))
        return KDA_ERR_CUDA;
    const int sms = max(1, sm_count());
    bwd_masks_kernel<<<unsigned(ceil_div(n_chunks, 8)), 256, 0, stream>>>(
        seg, N, RowStartTest::make(T_len), n_chunks, H, ws);
    if (cudaGetLastError() != cudaSuccess) return KDA_ERR_CUDA;
    // a chain is cut into pieces of kPiece chunks when it is longer than two of them
    bwd_chains_kernel<<<1, kChainThreads, 0, stream>>>(n_chunks, H, 2 * kPiece, ws);
    if (cudaGetLastError() != cudaSuccess) return KDA_ERR_CUDA;
    if (dynamic_smem_attr<scan_kernel<false>>(int(kScanSmem)) != cudaSuccess ||
        dynamic_smem_attr<scan_kernel<true>>(int(kScanSmem)) != cudaSuccess)
        return KDA_ERR_CUDA;
    ScanParams sp;
    sp.beta = static_cast<const __nv_bfloat16*>(beta);
    sp.scale = scale;
    sp.N = N;
    sp.H = H;
    sp.n_chunks = n_chunks;
    sp.ws = ws;
    sp.status = status_dev;
    const int64_t n_items = n_chunks * H;
    const unsigned scan_grid = unsigned(n_items < 2 * sms ? n_items : 2 * sms);
    const unsigned comb_grid = unsigned(4 * sms);
    // each direction: the pieces' end states, the combine, then the export pass
    for (int dn = 0; dn < 2; ++dn) {
        for (int phase = 1; phase >= 0; --phase) {
            sp.phase = phase;
            if (dn == 0)
                scan_kernel<false><<<scan_grid, kScanThreads, kScanSmem, stream>>>(m[1], m[2], m[3], sp);
            else
                scan_kernel<true><<<scan_grid, kScanThreads, kScanSmem, stream>>>(m[0], m[2], m[4], sp);
            if (cudaGetLastError() != cudaSuccess) return KDA_ERR_CUDA;
            if (phase == 1) {
                combine_kernel<<<comb_grid, 256, 0, stream>>>(n_chunks, H, dn, ws);
                if (cudaGetLastError() != cudaSuccess) return KDA_ERR_CUDA;
            }
        }
    }
    GradParams gp;
    gp.q = static_cast<const __nv_bfloat16*>(q);
    gp.k = static_cast<const __nv_bfloat16*>(k);
    gp.g = static_cast<const __nv_bfloat16*>(g);
    gp.beta = sp.beta;
    gp.scale = scale;
    gp.N = N;
    gp.H = H;
    gp.n_chunks = n_chunks;
    gp.ws = ws;
    gp.dq = dq;
    gp.dk = dk;
    gp.dv = dv;
    gp.dg = dg;
    gp.dbeta = dbeta;
    gp.status = status_dev;
    const unsigned grid = unsigned(n_items < sms ? n_items : sms);
    if (grad_dtype == KDA_F32) {
        if (dynamic_smem_attr<grad_kernel<float>>(int(kGradSmem)) != cudaSuccess) return KDA_ERR_CUDA;
        grad_kernel<float><<<grid, kGradThreads, kGradSmem, stream>>>(m[0], m[1], m[2], m[3], m[4], gp);
    } else {
        if (dynamic_smem_attr<grad_kernel<__nv_bfloat16>>(int(kGradSmem)) != cudaSuccess)
            return KDA_ERR_CUDA;
        grad_kernel<__nv_bfloat16><<<grid, kGradThreads, kGradSmem, stream>>>(m[0], m[1], m[2], m[3],
                                                                             m[4], gp);
    }
    if (cudaGetLastError() != cudaSuccess) return KDA_ERR_CUDA;
    // the items outside the factorised form's range, if any, in fp32
    RedoParams rp;
    rp.q = static_cast<const __nv_bfloat16*>(q);
    rp.k = gp.k;
    rp.v = static_cast<const __nv_bfloat16*>(v);
    rp.g = gp.g;
    rp.beta = gp.beta;
    rp.d_o = static_cast<const __nv_bfloat16*>(d_o);
    rp.scale = scale;
    rp.N = N;
    rp.H = H;
    rp.n_chunks = n_chunks;
    rp.ws = ws;
    rp.dq = dq;
    rp.dk = dk;
    rp.dv = dv;
    rp.dg = dg;
    rp.dbeta = dbeta;
    if (grad_dtype == KDA_F32) {
        if (dynamic_smem_attr<redo_kernel<float>>(int(kRedoSmem)) != cudaSuccess) return KDA_ERR_CUDA;
        redo_kernel<float><<<grid, kRedoThreads, kRedoSmem, stream>>>(rp);
    } else {
        if (dynamic_smem_attr<redo_kernel<__nv_bfloat16>>(int(kRedoSmem)) != cudaSuccess)
            return KDA_ERR_CUDA;
        redo_kernel<__nv_bfloat16><<<grid, kRedoThreads, kRedoSmem, stream>>>(rp);
    }
    return launch_status();
}

}  // namespace kda
