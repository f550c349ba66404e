// Parity oracle for the MoE expert-grouped token reorder.
//
// TEST INFRASTRUCTURE ONLY. This file is a plain, slow, single-threaded CPU
// restatement of what the operations compute: the FFN-worker batching (from
// flat arrays or a ScheduleContext, optionally over the whole tail), the
// routing-map permute and unpermute, and MoeUpdateExpert. Only the test suite, the
// smoke check and the benchmark's CPU-baseline leg may load it; the product
// path (the CUDA library and its Python binding) never does. It shares no code,
// header, table or helper with the CUDA path.
//
// Sources (web pages, cited by title and section):
//   [FWB]  "aclnnFfnWorkerBatching" (CANN ops-transformer docs): 功能说明 (the
//          four steps and the 计算公式), 参数说明 (parameter table),
//          约束说明 (constraints), 调用示例 (example program).
//   [UNP]  "MoeTokenUnpermuteWithRoutingMap 算子全解析" (CANN ops-transformer
//          article): 功能说明与计算公式 (derived sizes and the four branches),
//          参数说明 / 补充说明 (shapes and ranges), Kernel 实现 (pad kernel
//          prob lookup, IsValidInputIndex, prob != 0 skip, fp32 Cast/Muls/Add,
//          CAST_RINT).
//   [UPD]  "MoeUpdateExpert" (CANN ops-transformer README): 功能说明,
//          参数说明 and 约束说明.
//
// Where the pages are silent or garbled, the reading taken is stated at each
// use below.
//
// Floating point: the pages fix the arithmetic of the reduction (operands cast
// to fp32, multiply by the prob, add, one final cast with round-to-nearest-
// even), so this oracle computes in fp32 exactly that way, one rounded multiply
// and one rounded add per term. Build with -ffp-contract=off so the compiler
// does not fuse them.
//
// Build: g++ -O2 -std=c++17 -ffp-contract=off -fPIC -shared oracle.cpp

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <numeric>
#include <vector>

namespace {

// dtype codes shared by both operations' parameter tables.
enum : int32_t { DT_F16 = 0, DT_BF16 = 1, DT_INT8 = 2, DT_F32 = 3 };

// ---------------------------------------------------------------------------
// Scalar conversions, written from the IEEE-754 binary16 / bfloat16 formats.
// ---------------------------------------------------------------------------

float bits_to_float(uint32_t u) {
    float f;
    std::memcpy(&f, &u, 4);
    return f;
}

uint32_t float_to_bits(float f) {
    uint32_t u;
    std::memcpy(&u, &f, 4);
    return u;
}

// binary16 -> binary32 (exact).
float half_to_float(uint16_t h) {
    const uint32_t sign = (uint32_t)(h >> 15) << 31;
    const int exp = (h >> 10) & 0x1f;
    const uint32_t man = h & 0x3ff;
    if (exp == 0x1f) {  // inf / nan
        return bits_to_float(sign | 0x7f800000u | (man << 13) | (man ? 0x00400000u : 0u));
    }
    if (exp == 0) {  // zero or subnormal: value = man * 2^-24
        float v = (float)man * (1.0f / 16777216.0f);
        return sign ? -v : v;
    }
    return bits_to_float(sign | ((uint32_t)(exp - 15 + 127) << 23) | (man << 13));
}

// binary32 -> binary16, round to nearest, ties to even.
uint16_t float_to_half(float f) {
    const uint32_t u = float_to_bits(f);
    const uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    const int exp = (int)((u >> 23) & 0xff);
    uint32_t man = u & 0x7fffffu;
    if (exp == 0xff) {  // inf / nan (keep nan quiet)
        return (uint16_t)(sign | 0x7c00u | (man ? 0x200u | (man >> 13) : 0u));
    }
    const int e = exp - 127;  // unbiased exponent
    if (e > 15) return (uint16_t)(sign | 0x7c00u);  // overflow -> inf
    if (e >= -14) {
        // normal half: keep 10 mantissa bits, round the 13 dropped bits
        uint32_t keep = man >> 13;
        uint32_t rest = man & 0x1fffu;
        uint32_t he = (uint32_t)(e + 15);
        uint32_t r = (he << 10) | keep;
        if (rest > 0x1000u || (rest == 0x1000u && (keep & 1u))) r += 1;  // may carry into exponent / inf
        return (uint16_t)(sign | r);
    }
    // subnormal half (or underflow to zero): value = m * 2^-24 with m < 1024
    if (e < -25) return sign;  // below half of the smallest subnormal
    man |= 0x800000u;  // implicit one, value = man * 2^(e-23)
    const int shift = (-14 - e) + 13;  // bits to drop so the unit is 2^-24
    uint32_t keep = man >> shift;
    uint32_t rest = man & ((1u << shift) - 1u);
    uint32_t half = 1u << (shift - 1);
    if (rest > half || (rest == half && (keep & 1u))) keep += 1;
    return (uint16_t)(sign | keep);
}

float bf16_to_float(uint16_t b) { return bits_to_float((uint32_t)b << 16); }

// binary32 -> bfloat16, round to nearest, ties to even.
uint16_t float_to_bf16(float f) {
    const uint32_t u = float_to_bits(f);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x7fffffu)) {  // nan: keep quiet
        return (uint16_t)((u >> 16) | 0x40u);
    }
    uint32_t keep = u >> 16;
    uint32_t rest = u & 0xffffu;
    if (rest > 0x8000u || (rest == 0x8000u && (keep & 1u))) keep += 1;
    return (uint16_t)keep;
}

size_t elem_bytes(int32_t dt) {
    switch (dt) {
        case DT_F16: return 2;
        case DT_BF16: return 2;
        case DT_INT8: return 1;
        case DT_F32: return 4;
    }
    return 0;
}

float load_as_float(const void* base, int64_t index, int32_t dt) {
    const uint8_t* p = (const uint8_t*)base + (size_t)index * elem_bytes(dt);
    if (dt == DT_F32) {
        float f;
        std::memcpy(&f, p, 4);
        return f;
    }
    uint16_t h;
    std::memcpy(&h, p, 2);
    return dt == DT_F16 ? half_to_float(h) : bf16_to_float(h);
}

void store_from_float(void* base, int64_t index, int32_t dt, float v) {
    uint8_t* p = (uint8_t*)base + (size_t)index * elem_bytes(dt);
    if (dt == DT_F32) {
        std::memcpy(p, &v, 4);
        return;
    }
    uint16_t h = dt == DT_F16 ? float_to_half(v) : float_to_bf16(v);
    std::memcpy(p, &h, 2);
}

// Copy one element of dtype dt without interpreting it (the prob outputs keep
// the probs dtype bit for bit).
void copy_elem(void* dst, int64_t di, const void* src, int64_t si, int32_t dt) {
    const size_t b = elem_bytes(dt);
    std::memcpy((uint8_t*)dst + (size_t)di * b, (const uint8_t*)src + (size_t)si * b, b);
}

}  // namespace

extern "C" {

// Array conversions, exported so the tests can pin the scalar routines against
// numpy / torch conversions.
void oracle_half_to_float(const uint16_t* in, float* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = half_to_float(in[i]);
}
void oracle_float_to_half(const float* in, uint16_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = float_to_half(in[i]);
}
void oracle_bf16_to_float(const uint16_t* in, float* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = bf16_to_float(in[i]);
}
void oracle_float_to_bf16(const float* in, uint16_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = float_to_bf16(in[i]);
}

// ---------------------------------------------------------------------------
// FFN-worker batching  [FWB 功能说明 steps 2-4, 计算公式, 参数说明]
//
//   gather_idx, _ = sort(expert_ids_in)           (masked slots keyed large)
//   y[i]          = token_data[gather_idx[i]]     (+ dynamic scale in INT8 mode)
//   group_list[e] = [expert_id_e, expert_token_num_e]
//   actual_token_num = sum_e expert_token_num_e
//
// Readings:
//  * Y = A * BS * (topK+1)   (maxOutShape row of 参数说明).
//  * key(s) = layer_id * E_l + expert_ids[s] when 0 <= expert_ids[s] < E_l,
//    else the sentinel E (masked). E_l = expertNum / max(layerNum, 1).
//  * The sort is stable: ties keep slot order.
//  * group_list is compacted: row r = [key, count] of the r-th distinct
//    unmasked key in ascending order, remaining rows [0, 0].
//  * expertOffsets[i] = i - (first output index of i's key).
//  * tokenIds[i] = token_in[g] if token_in is given, else g (the slot index).
//  * Rows i >= U (masked tail): y and dynamicScale are left untouched; the
//    four int32 id outputs are -1.
//  * INT8: row = H int8 bytes; the fp32 scale is read from scales_base +
//    g*scale_stride if scales_base is given, else right after the row data
//    (token_data + g*row_stride + H).
//  * sorted_indices_out (optional): for each slot s its output row, -1 if
//    masked: the inverse of gather_idx, i.e. the sortedIndices that the
//    unpermute of page [UNP] takes in its non-padded layout.
//
// Returns 0 on success, nonzero on a shape it cannot handle.
// ---------------------------------------------------------------------------
int oracle_batching(const int32_t* expert_ids, int32_t layer_id, const uint8_t* token_data,
                    int64_t row_stride, const uint8_t* scales_base, int64_t scale_stride,
                    const int32_t* session_in, const int32_t* micro_in, const int32_t* token_in,
                    int64_t expertNum, int64_t A, int64_t BS, int64_t K1, int64_t H,
                    int64_t tokenDtype, int64_t layerNum, uint8_t* y, int64_t* group_list,
                    int32_t* session_out, int32_t* micro_out, int32_t* token_out,
                    int32_t* expert_offsets, float* dynamic_scale, int64_t* actual_token_num,
                    int32_t* sorted_indices_out, int32_t* gather_idx_out, int32_t full_tail) {
    if (expertNum <= 0 || A <= 0 || BS <= 0 || K1 <= 0 || H <= 0) return 1;
    if (tokenDtype != DT_F16 && tokenDtype != DT_BF16 && tokenDtype != DT_INT8) return 2;
    const int64_t Y = A * BS * K1;
    const int64_t E = expertNum;
    const int64_t L = layerNum > 0 ? layerNum : 1;
    if (E % L != 0) return 3;
    const int64_t El = E / L;
    if (layer_id < 0 || layer_id >= L) return 4;
    const int64_t row_bytes = H * (int64_t)elem_bytes((int32_t)tokenDtype);

    // key of every slot; masked slots get the large value E
    std::vector<int64_t> key(Y);
    for (int64_t s = 0; s < Y; ++s) {
        const int64_t id = expert_ids[s];
        key[s] = (id >= 0 && id < El) ? (int64_t)layer_id * El + id : E;
    }

    // gather_idx = stable sort of the slots by key
    std::vector<int64_t> gather_idx(Y);
    std::iota(gather_idx.begin(), gather_idx.end(), (int64_t)0);
    std::stable_sort(gather_idx.begin(), gather_idx.end(),
                     [&](int64_t a, int64_t b) { return key[a] < key[b]; });

    int64_t U = 0;
    for (int64_t s = 0; s < Y; ++s) U += key[s] < E ? 1 : 0;

    // y[i] = token_data[gather_idx[i]] for the unmasked prefix (every row
    // when the formula is applied to the masked tail too)
    const int64_t gathered = full_tail ? Y : U;
    for (int64_t i = 0; i < gathered; ++i) {
        const int64_t g = gather_idx[i];
        std::memcpy(y + (size_t)(i * row_bytes), token_data + (size_t)(g * row_stride),
                    (size_t)row_bytes);
        if (tokenDtype == DT_INT8) {
            const uint8_t* sp = scales_base ? scales_base + (size_t)(g * scale_stride)
                                            : token_data + (size_t)(g * row_stride + H);
            std::memcpy(&dynamic_scale[i], sp, 4);
        }
    }

    // id lookups and the offset inside the expert group
    int64_t group_start = 0;
    for (int64_t i = 0; i < Y; ++i) {
        const int64_t g = gather_idx[i];
        if (i < U) {
            if (i == 0 || key[gather_idx[i - 1]] != key[g]) group_start = i;
            session_out[i] = session_in[g];
            micro_out[i] = micro_in[g];
            token_out[i] = token_in ? token_in[g] : (int32_t)g;
            expert_offsets[i] = (int32_t)(i - group_start);
        } else if (full_tail) {
            // a masked slot's own ids; it belongs to no expert group
            session_out[i] = session_in[g];
            micro_out[i] = micro_in[g];
            token_out[i] = token_in ? token_in[g] : (int32_t)g;
            expert_offsets[i] = -1;
        } else {
            session_out[i] = -1;
            micro_out[i] = -1;
            token_out[i] = -1;
            expert_offsets[i] = -1;
        }
    }

    // group_list: one row per change point of the sorted keys, then [0, 0]
    int64_t rows = 0;
    for (int64_t i = 0; i < U; ++i) {
        const int64_t k = key[gather_idx[i]];
        if (i == 0 || key[gather_idx[i - 1]] != k) {
            group_list[2 * rows + 0] = k;
            group_list[2 * rows + 1] = 0;
            ++rows;
        }
        group_list[2 * (rows - 1) + 1] += 1;
    }
    for (int64_t r = rows; r < E; ++r) {
        group_list[2 * r + 0] = 0;
        group_list[2 * r + 1] = 0;
    }

    // actual_token_num = sum of the expert token counts
    int64_t total = 0;
    for (int64_t r = 0; r < rows; ++r) total += group_list[2 * r + 1];
    actual_token_num[0] = total;

    if (sorted_indices_out) {
        for (int64_t s = 0; s < Y; ++s) sorted_indices_out[s] = -1;
        for (int64_t i = 0; i < U; ++i) sorted_indices_out[gather_idx[i]] = (int32_t)i;
    }
    if (gather_idx_out) {
        for (int64_t i = 0; i < Y; ++i) gather_idx_out[i] = (int32_t)gather_idx[i];
    }
    return 0;
}

// ---------------------------------------------------------------------------
// FFN-worker batching from a ScheduleContext  [FWB 功能说明 step 1, the
// ScheduleContext / FfnDataDesc structs and the token_info / token_data fill
// of 调用示例]
//
// The 1024-byte packed context: CommonArea at byte 0 (u32 session_num,
// micro_batch_num, micro_batch_size, selected_expert_num, expert_num, ...),
// ControlArea at 128, AttentionArea at 256, FfnArea at 384 (u64
// token_info_buf, token_info_buf_size, token_data_buf, token_data_buf_size,
// ...). token_info_buf holds one FfnDataDesc per (session, micro-batch) block,
// sessions outer: i32 flag, i32 layer_id, then micro_batch_size *
// selected_expert_num i32 expert ids. token_data_buf holds one row per slot in
// the same order.
//
// Readings:
//  * The slots are the blocks' expert ids in block order; slot g of block b
//    has session id b / micro_batch_num, micro-batch id b % micro_batch_num
//    and token id g.
//  * Each block carries its own layer_id: key = layer_id * E_l + id; a block
//    whose layer_id is outside [0, max(layerNum,1)) has all its slots masked.
//  * needSchedule = 1: a block takes part only if its flag is 1 (ready);
//    otherwise all its slots are masked. needSchedule = 0 ignores the flags.
//    `status` = number of blocks not ready (0 with needSchedule = 0).
//  * The context is invalid when a count is 0, the context's slots exceed
//    Y = A*BS*(topK+1) of maxOutShape, expert_num != E_l, or a buffer is
//    NULL or too small, or token_info_buf is not 4-byte aligned (its fields
//    are int32): then every slot is masked and status = -1.
//  * Outputs are sized for Y rows; rows past the context's slots belong to
//    the masked tail (ids -1, y untouched).
//  * full_tail: the formulas of 计算公式 are applied to the masked rows too,
//    as far as they have a slot in token_data_buf: y, the scale, session,
//    micro-batch and token ids of the slot; expertOffsets stays -1.
// The host copies of token_info_buf / token_data_buf are passed separately
// (the context itself holds device addresses).
// ---------------------------------------------------------------------------
int oracle_batching_context(const uint8_t* ctx, const uint8_t* token_info,
                            const uint8_t* token_data, int64_t expertNum, int64_t A, int64_t BS,
                            int64_t K1, int64_t H, int64_t tokenDtype, int64_t needSchedule,
                            int64_t layerNum, uint8_t* y, int64_t* group_list,
                            int32_t* session_out, int32_t* micro_out, int32_t* token_out,
                            int32_t* expert_offsets, float* dynamic_scale,
                            int64_t* actual_token_num, int32_t* status, int32_t full_tail) {
    if (expertNum <= 0 || A <= 0 || BS <= 0 || K1 <= 0 || H <= 0) return 1;
    const int64_t Y = A * BS * K1;
    const int64_t E = expertNum;
    const int64_t L = layerNum > 0 ? layerNum : 1;
    if (E % L != 0) return 3;
    const int64_t El = E / L;
    const int64_t es = (int64_t)elem_bytes((int32_t)tokenDtype);
    const int64_t row_bytes = H * es;
    const int64_t row_stride = row_bytes + (tokenDtype == DT_INT8 ? 4 : 0);

    uint32_t common[5];
    std::memcpy(common, ctx, sizeof(common));
    const int64_t sessions = common[0], micro = common[1], mbs = common[2], sel = common[3];
    const int64_t expert_num_ctx = common[4];
    uint64_t ffn[4];
    std::memcpy(ffn, ctx + 384, sizeof(ffn));  // info buf, info size, data buf, data size
    const int64_t per_block = mbs * sel;
    const int64_t blocks = sessions * micro;
    const int64_t slots = blocks * per_block;
    const int64_t block_bytes = 8 + 4 * per_block;
    bool valid = sessions > 0 && micro > 0 && mbs > 0 && sel > 0 && slots <= Y &&
                 expert_num_ctx == El && ffn[0] != 0 && ffn[2] != 0 && (ffn[0] & 3u) == 0 &&
                 (int64_t)ffn[1] >= blocks * block_bytes && (int64_t)ffn[3] >= slots * row_stride;

    std::vector<int64_t> key(Y, E);
    std::vector<int32_t> sess(Y, 0), mb(Y, 0);
    int32_t not_ready = 0;
    if (valid) {
        for (int64_t b = 0; b < blocks; ++b) {
            const uint8_t* desc = token_info + b * block_bytes;
            int32_t flag, layer;
            std::memcpy(&flag, desc, 4);
            std::memcpy(&layer, desc + 4, 4);
            const bool ready = needSchedule == 0 || flag == 1;
            if (!ready) ++not_ready;
            for (int64_t j = 0; j < per_block; ++j) {
                const int64_t g = b * per_block + j;
                int32_t id;
                std::memcpy(&id, desc + 8 + 4 * j, 4);
                if (ready && layer >= 0 && layer < L && id >= 0 && id < El) key[g] = layer * El + id;
                sess[g] = (int32_t)(b / micro);
                mb[g] = (int32_t)(b % micro);
            }
        }
    }
    if (status) status[0] = valid ? not_ready : -1;

    std::vector<int64_t> gather_idx(Y);
    std::iota(gather_idx.begin(), gather_idx.end(), (int64_t)0);
    std::stable_sort(gather_idx.begin(), gather_idx.end(),
                     [&](int64_t a, int64_t b) { return key[a] < key[b]; });
    int64_t U = 0;
    for (int64_t s = 0; s < Y; ++s) U += key[s] < E ? 1 : 0;
    // slots with a row in token_data_buf (none when the context is invalid)
    const int64_t n_src = valid ? slots : 0;
    for (int64_t i = 0; i < Y; ++i) {
        const int64_t g = gather_idx[i];
        if (!(i < U || (full_tail && g < n_src))) continue;
        std::memcpy(y + i * row_bytes, token_data + g * row_stride, (size_t)row_bytes);
        if (tokenDtype == DT_INT8) std::memcpy(&dynamic_scale[i], token_data + g * row_stride + row_bytes, 4);
    }
    int64_t group_start = 0;
    for (int64_t i = 0; i < Y; ++i) {
        const int64_t g = gather_idx[i];
        if (i < U) {
            if (i == 0 || key[gather_idx[i - 1]] != key[g]) group_start = i;
            session_out[i] = sess[g];
            micro_out[i] = mb[g];
            token_out[i] = (int32_t)g;
            expert_offsets[i] = (int32_t)(i - group_start);
        } else if (full_tail && g < n_src) {
            session_out[i] = sess[g];
            micro_out[i] = mb[g];
            token_out[i] = (int32_t)g;
            expert_offsets[i] = -1;
        } else {
            session_out[i] = micro_out[i] = token_out[i] = expert_offsets[i] = -1;
        }
    }
    int64_t rows = 0;
    for (int64_t i = 0; i < U; ++i) {
        const int64_t k = key[gather_idx[i]];
        if (i == 0 || key[gather_idx[i - 1]] != k) {
            group_list[2 * rows] = k;
            group_list[2 * rows + 1] = 0;
            ++rows;
        }
        group_list[2 * (rows - 1) + 1] += 1;
    }
    for (int64_t r = rows; r < E; ++r) group_list[2 * r] = group_list[2 * r + 1] = 0;
    actual_token_num[0] = U;
    return 0;
}

// ---------------------------------------------------------------------------
// Routing-map permute  [UNP 算子定位: the permute step that precedes the
// unpermute rearranges the tokens by routingMap into an expert-grouped compact
// layout, permutedTokens, so that each expert reads its tokens contiguously]
//
// Readings, chosen so that the unpermute takes these outputs:
//  * Not padded: the rows are the (token, expert) pairs with routingMap = 1 in
//    expert-major order (expert ascending, then token ascending): the order of
//    probs.T.maskedSelect(routingMap.T). permutedTokens[r] = tokens[t(r)] for
//    r < topK*T. sortedIndices[t*topK + j] = row of t's j-th routed expert
//    (ascending expert id), -1 for j >= its count; a pair whose row is not
//    below topK*T gets -1 too. rows_out = min(pairs, topK*T).
//  * Padded (capacity layout): expert e keeps its first `capacity` routed
//    tokens (ascending token id) in rows e*capacity + r; sortedIndices of those
//    rows = the token id; the remaining rows are padding: sortedIndices -1 and
//    a zero row. rows_out = rows kept.
// ---------------------------------------------------------------------------
int oracle_permute(const void* tokens, const int8_t* routingMap, int64_t T, int64_t H,
                   int32_t tokenDtype, int64_t Eu, int64_t topK, int32_t padded, int64_t capacity,
                   void* permuted, int32_t* sortedIndices, int32_t* rows_out) {
    if (T <= 0 || H <= 0 || Eu <= 0) return 1;
    const size_t row_bytes = (size_t)H * elem_bytes(tokenDtype);
    const uint8_t* src = (const uint8_t*)tokens;
    uint8_t* dst = (uint8_t*)permuted;
    if (!padded) {
        if (topK <= 0) return 2;
        const int64_t n = T * topK;
        // rows in expert-major order
        std::vector<int64_t> row_of((size_t)(T * Eu), -1);
        int64_t r = 0;
        for (int64_t e = 0; e < Eu; ++e) {
            for (int64_t t = 0; t < T; ++t) {
                if (routingMap[t * Eu + e] != 0) {
                    row_of[(size_t)(t * Eu + e)] = r;
                    if (r < n) std::memcpy(dst + (size_t)r * row_bytes, src + (size_t)t * row_bytes, row_bytes);
                    ++r;
                }
            }
        }
        for (int64_t t = 0; t < T; ++t) {
            int64_t j = 0;
            for (int64_t e = 0; e < Eu; ++e) {
                const int64_t ro = row_of[(size_t)(t * Eu + e)];
                if (ro < 0) continue;
                if (j < topK) sortedIndices[t * topK + j] = ro < n ? (int32_t)ro : -1;
                ++j;
            }
            for (; j < topK; ++j) sortedIndices[t * topK + j] = -1;
        }
        rows_out[0] = (int32_t)(r < n ? r : n);
    } else {
        if (capacity <= 0) return 3;
        int64_t kept = 0;
        for (int64_t e = 0; e < Eu; ++e) {
            int64_t r = 0;
            for (int64_t t = 0; t < T; ++t) {
                if (routingMap[t * Eu + e] != 0 && r < capacity) {
                    sortedIndices[e * capacity + r] = (int32_t)t;
                    std::memcpy(dst + (size_t)(e * capacity + r) * row_bytes, src + (size_t)t * row_bytes, row_bytes);
                    ++r;
                }
            }
            kept += r;
            for (; r < capacity; ++r) {
                sortedIndices[e * capacity + r] = -1;
                std::memset(dst + (size_t)(e * capacity + r) * row_bytes, 0, row_bytes);
            }
        }
        rows_out[0] = (int32_t)kept;
    }
    return 0;
}

// ---------------------------------------------------------------------------
// Logical -> physical expert mapping with pruning  [UPD 功能说明, 参数说明]
//
// eplbTable [moeExpertNum, F] int32: column 0 = the number of instances
// `count` of the row's logical expert, columns 1..count = their instance ids.
//
// Readings:
//  * balancedExpertIds[b, k] = eplbTable[e, 1 + c] with e = expertIds[b, k]
//    and c = localRankId % count (balanceMode 0, by rank) or b % count
//    (balanceMode 1, by token); -1 when e is outside [0, moeExpertNum) or
//    count is outside [1, F - 1]. The page names the two modes but gives no
//    rule for which instance: parity unpinned beyond the result being one of
//    the expert's instances (and the same for every token of a rank in
//    mode 0, cycling over the tokens in mode 1).
//  * With scales and thresholds: balancedActiveMask[b, k] = the token is
//    active (activeMask[b], all active if not given) and not
//    f32(scale[b, k]) < threshold[k] (pruned when below; equal and NaN are
//    kept). Without them the mask is not written.
//  * expertIds and the output are int32 (idBytes 4) or int64 (idBytes 8).
// ---------------------------------------------------------------------------
int oracle_update_expert(const void* expertIds, int32_t idBytes, const int32_t* table,
                         const void* scales, int32_t scalesDtype, const float* threshold,
                         const uint8_t* activeMask, int64_t BS, int64_t K, int64_t moeExpertNum,
                         int64_t F, int64_t localRankId, int64_t balanceMode, void* balancedIds,
                         uint8_t* balancedMask) {
    if (BS <= 0 || K <= 0 || moeExpertNum <= 0 || F < 2) return 1;
    for (int64_t b = 0; b < BS; ++b) {
        for (int64_t k = 0; k < K; ++k) {
            const int64_t i = b * K + k;
            int64_t e;
            if (idBytes == 8) {
                int64_t v;
                std::memcpy(&v, (const uint8_t*)expertIds + 8 * i, 8);
                e = v;
            } else {
                int32_t v;
                std::memcpy(&v, (const uint8_t*)expertIds + 4 * i, 4);
                e = v;
            }
            int64_t out = -1;
            if (e >= 0 && e < moeExpertNum) {
                const int64_t count = table[e * F];
                if (count >= 1 && count <= F - 1) {
                    const int64_t c = (balanceMode == 0 ? localRankId : b) % count;
                    out = table[e * F + 1 + c];
                }
            }
            if (idBytes == 8) {
                std::memcpy((uint8_t*)balancedIds + 8 * i, &out, 8);
            } else {
                const int32_t o = (int32_t)out;
                std::memcpy((uint8_t*)balancedIds + 4 * i, &o, 4);
            }
            if (scales && threshold && balancedMask) {
                const bool active = activeMask ? activeMask[b] != 0 : true;
                const float sc = load_as_float(scales, i, scalesDtype);
                balancedMask[i] = (active && !(sc < threshold[k])) ? 1 : 0;
            }
        }
    }
    return 0;
}

// ---------------------------------------------------------------------------
// Routing-map unpermute  [UNP 功能说明与计算公式 branches (1)-(4)]
//
// Derived sizes: topK_num = permutedRows // numTokens, capacity =
// n // numExperts (padded), with n = len(sortedIndices).
//
// (1) probs, padded:   permuteProbs[i] = probs[sortedIndices[i], i // capacity]
//                      permuteTokenId, outIndex = sortedIndices.sort()
//                      out[permuteTokenId[i]] += permuted[outIndex[i]] * permuteProbs[outIndex[i]]
// (2) probs, !padded:  permuteProbs = probs.T.maskedSelect(routingMap.T)
//                      if sortedIndices[i] valid: out[i // topK] += permuted[sortedIndices[i]] * permuteProbs[i]
// (3) no probs, padded:   as (1) without the weight
// (4) no probs, !padded:  as (2) without the weight
//
// Readings:
//  * "+=" accumulates (the page's text says 累加求和 throughout).
//  * One multiplication per term, by the slot's (2) or the row's (1) prob.
//  * A term is skipped unless its index is valid (IsValidInputIndex) and, with
//    probs, its prob != 0 (the non-pad kernel's prob_value != 0 test).
//    Valid means 0 <= idx < permutedRows when not padded, 0 <= idx < numTokens
//    when padded.
//  * Arithmetic: fp32 accumulator starting at 0, term = f32(x) * f32(p)
//    rounded to fp32, added in ascending slot (not padded) / ascending row
//    (padded) order, one final round-to-nearest-even cast to the token dtype.
//  * The sorts are stable. Not padded: outIndex = stable ascending argsort of
//    sortedIndices with every invalid entry first; permuteTokenId =
//    outIndex // topK. Padded: invalid entries sort last; permuteTokenId =
//    the sorted values themselves.
//  * permuteProbs (not padded): the maskedSelect result, truncated to n and
//    zero-filled after its last element. Padded, invalid index: 0.
//  * Without probs, permuteProbs is not written.
// ---------------------------------------------------------------------------
int oracle_unpermute(const void* permuted, const int32_t* sortedIndices, const int8_t* routingMap,
                     const void* probs, int64_t permutedRows, int64_t H, int32_t tokenDtype,
                     int64_t n, int32_t probsDtype, int64_t T, int64_t Eu, int32_t padded,
                     void* out, int32_t* outIndex, int32_t* permuteTokenId, void* permuteProbs) {
    if (T <= 0 || H <= 0 || permutedRows < 0 || n < 0) return 1;
    const bool has_probs = probs != nullptr;
    const int64_t topK = permutedRows / T;

    // permuteProbs
    std::vector<float> weight(has_probs ? n : 0, 0.0f);
    if (has_probs && !padded) {
        // probs.T.maskedSelect(routingMap.T): walk the transposed matrices in
        // row-major order, i.e. expert by expert, token by token.
        int64_t pos = 0;
        for (int64_t e = 0; e < Eu; ++e) {
            for (int64_t t = 0; t < T; ++t) {
                if (routingMap[t * Eu + e] != 0) {
                    if (pos < n) copy_elem(permuteProbs, pos, probs, t * Eu + e, probsDtype);
                    ++pos;
                }
            }
        }
        for (int64_t i = pos; i < n; ++i) store_from_float(permuteProbs, i, probsDtype, 0.0f);
    } else if (has_probs && padded) {
        if (Eu <= 0) return 2;
        const int64_t capacity = n / Eu;
        if (capacity <= 0) return 3;
        for (int64_t i = 0; i < n; ++i) {
            const int64_t v = sortedIndices[i];
            if (v >= 0 && v < T) {
                copy_elem(permuteProbs, i, probs, v * Eu + i / capacity, probsDtype);
            } else {
                store_from_float(permuteProbs, i, probsDtype, 0.0f);
            }
        }
    }
    if (has_probs) {
        for (int64_t i = 0; i < n; ++i) weight[i] = load_as_float(permuteProbs, i, probsDtype);
    }

    // sort of sortedIndices -> outIndex (positions), permuteTokenId
    std::vector<int64_t> sort_key(n);
    for (int64_t i = 0; i < n; ++i) {
        const int64_t v = sortedIndices[i];
        if (padded) {
            sort_key[i] = (v >= 0 && v < T) ? v : T;  // invalid last
        } else {
            sort_key[i] = (v >= 0 && v < permutedRows) ? v : -1;  // invalid first
        }
    }
    std::vector<int64_t> order(n);
    std::iota(order.begin(), order.end(), (int64_t)0);
    std::stable_sort(order.begin(), order.end(),
                     [&](int64_t a, int64_t b) { return sort_key[a] < sort_key[b]; });
    for (int64_t i = 0; i < n; ++i) {
        outIndex[i] = (int32_t)order[i];
        permuteTokenId[i] = padded ? sortedIndices[order[i]] : (int32_t)(order[i] / topK);
    }

    // accumulate in fp32
    std::vector<float> acc((size_t)(T * H), 0.0f);
    if (!padded) {
        for (int64_t i = 0; i < n; ++i) {
            const int64_t v = sortedIndices[i];
            if (v < 0 || v >= permutedRows) continue;
            const int64_t t = i / topK;
            if (t >= T) continue;
            float p = 1.0f;
            if (has_probs) {
                p = weight[i];
                if (p == 0.0f) continue;
            }
            for (int64_t h = 0; h < H; ++h) {
                const float x = load_as_float(permuted, v * H + h, tokenDtype);
                float term = x;
                if (has_probs) term = x * p;
                acc[(size_t)(t * H + h)] = acc[(size_t)(t * H + h)] + term;
            }
        }
    } else {
        for (int64_t i = 0; i < n; ++i) {
            const int64_t r = order[i];
            const int64_t t = sortedIndices[r];
            if (t < 0 || t >= T) continue;
            if (r >= permutedRows) continue;
            float p = 1.0f;
            if (has_probs) {
                p = weight[r];
                if (p == 0.0f) continue;
            }
            for (int64_t h = 0; h < H; ++h) {
                const float x = load_as_float(permuted, r * H + h, tokenDtype);
                float term = x;
                if (has_probs) term = x * p;
                acc[(size_t)(t * H + h)] = acc[(size_t)(t * H + h)] + term;
            }
        }
    }
    for (int64_t j = 0; j < T * H; ++j) store_from_float(out, j, tokenDtype, acc[(size_t)j]);
    return 0;
}

}  // extern "C"
