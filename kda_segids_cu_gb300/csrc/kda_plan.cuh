// kda_plan.cuh -- the chunk plan that the planner kernels of the bf16 path write into
// the caller's workspace, read by the chunk kernel and by the per-segment state pass.
#pragma once

#include "kda_common.cuh"

namespace kda {
namespace tc {

struct ChunkMeta {
    unsigned long long start;     // bit i: token i of the chunk starts a segment
    unsigned long long valid;     // bit i: token i exists and is not padding
};

struct Plan {                      // device view of the workspace
    int32_t* counters;             // [0] n_units, [1] next item, [2] n_chunks, [3] n_active,
                                   // [4] next unit of the state pass, [5] chunk-kernel CTAs
                                   // finished (the last one rewinds [1] and [5]), [6] units
                                   // the fast chunk kernel left to the safe one, [7] split
                                   // pieces with a successor (= slots used), [8] the state-only
                                   // phase's next item, [10] the fast kernel's call count (the
                                   // epoch of the slots' flags), [11] slots the workspace holds
    ChunkMeta* meta;               // [n_chunks]
    int32_t* first_cut;            // [n_chunks] first start-or-padding row, 64 if none
    int32_t* block_cut;            // [n_blocks]
    int32_t* cut_list;             // [n_chunks]
    int4* units;                   // [n_chunks] (c0, c1, row_lo, row_hi)
    int32_t* order;                // [n_chunks] unit indices, longest first
    int32_t* rank_base;            // [n_chunks] segment starts before the chunk (state calls only)
    int32_t* active;               // [n_chunks] chunks holding a start or a carried segment's end
                                   // (state calls only), in order
    int32_t* redo;                 // [n_chunks] positions (in order) of the units left to the
                                   // safe chunk kernel, counters[6] of them
    int32_t* redo_flag;            // [n_chunks] per position: 1 once listed in redo
    int4* units2;                  // [n_chunks] the units after splitting (then copied to units)
    int32_t* unit_in;              // [n_chunks] per unit: the slot holding the state it starts
                                   // from, or -1 (read only when counters[7] > 0)
    int4* apiece;                  // [n_chunks] pieces with a successor, by slot: (unit, slot of
                                   // the state it starts from or -1, slot it fills, 0)
};

// A long unit is split into pieces: leading pieces of at most kPieceChunks chunks and a last
// one. Slot s holds, per head, the state at the start of the piece after the s-th leading
// piece ([128][128] fp32, row = key channel) and a flag (the call's epoch + 1 once written).
constexpr int kPieceChunks = 64;
constexpr size_t kSlotStateBytes = size_t(128) * 128 * 4;

__host__ __device__ inline size_t slot_flags_bytes(int64_t max_slots, int32_t H) {
    return (size_t(max_slots) * H * 4 + 255) & ~size_t(255);
}

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

__host__ __device__ inline size_t plan_bytes(int64_t n_chunks) {
    size_t b = align256(64 * sizeof(int32_t));
    b += align256(n_chunks * sizeof(ChunkMeta));
    b += align256(n_chunks * sizeof(int32_t)) * 9;   // first_cut, block_cut, cut_list, order,
                                                     // rank_base, active, redo, redo_flag,
                                                     // unit_in
    b += align256(n_chunks * sizeof(int4)) * 3;      // units, units2, apiece
    return b;
}

// Slots that `bytes` past the plan hold for H heads.
__host__ __device__ inline int64_t slots_in(size_t bytes, int32_t H) {
    const size_t per = size_t(H) * (kSlotStateBytes + 4);
    if (bytes < 512 + per) return 0;
    return int64_t((bytes - 512) / per);
}

__host__ __device__ inline int32_t* slot_flags(void* ws, int64_t n_chunks) {
    return reinterpret_cast<int32_t*>(static_cast<uint8_t*>(ws) + plan_bytes(n_chunks));
}
__host__ __device__ inline float* slot_state(void* ws, int64_t n_chunks, int64_t max_slots,
                                             int32_t H, int64_t slot, int32_t h) {
    uint8_t* base = static_cast<uint8_t*>(ws) + plan_bytes(n_chunks) + slot_flags_bytes(max_slots, H);
    return reinterpret_cast<float*>(base + (size_t(slot) * H + h) * kSlotStateBytes);
}

__host__ __device__ inline Plan plan_view(void* ws, int64_t n_chunks) {
    uint8_t* p = static_cast<uint8_t*>(ws);
    Plan pl;
    pl.counters = reinterpret_cast<int32_t*>(p);      p += align256(64 * sizeof(int32_t));
    pl.meta = reinterpret_cast<ChunkMeta*>(p);        p += align256(n_chunks * sizeof(ChunkMeta));
    pl.first_cut = reinterpret_cast<int32_t*>(p);     p += align256(n_chunks * sizeof(int32_t));
    pl.block_cut = reinterpret_cast<int32_t*>(p);     p += align256(n_chunks * sizeof(int32_t));
    pl.cut_list = reinterpret_cast<int32_t*>(p);      p += align256(n_chunks * sizeof(int32_t));
    pl.order = reinterpret_cast<int32_t*>(p);         p += align256(n_chunks * sizeof(int32_t));
    pl.rank_base = reinterpret_cast<int32_t*>(p);     p += align256(n_chunks * sizeof(int32_t));
    pl.active = reinterpret_cast<int32_t*>(p);        p += align256(n_chunks * sizeof(int32_t));
    pl.redo = reinterpret_cast<int32_t*>(p);          p += align256(n_chunks * sizeof(int32_t));
    pl.redo_flag = reinterpret_cast<int32_t*>(p);     p += align256(n_chunks * sizeof(int32_t));
    pl.unit_in = reinterpret_cast<int32_t*>(p);       p += align256(n_chunks * sizeof(int32_t));
    pl.units2 = reinterpret_cast<int4*>(p);           p += align256(n_chunks * sizeof(int4));
    pl.apiece = reinterpret_cast<int4*>(p);           p += align256(n_chunks * sizeof(int4));
    pl.units = reinterpret_cast<int4*>(p);
    return pl;
}

}  // namespace tc
}  // namespace kda
