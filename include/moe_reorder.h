/*
 * moe_reorder.h -- C ABI of the GB300 MoE expert-grouped token reorder.
 *
 * Two operations, each a two-stage call in the style of the pages' aclnn
 * interfaces (a get-workspace-size call that validates and sizes, then an
 * execute call that enqueues on a stream):
 *
 *   ffnwb_batching  -- "aclnnFfnWorkerBatching": 功能说明 (steps 2-4 and the
 *                      计算公式), 参数说明 (parameter table), 约束说明.
 *   moe_unpermute   -- "MoeTokenUnpermuteWithRoutingMap 算子全解析":
 *                      功能说明与计算公式 (derived sizes, four branches),
 *                      参数说明 / 补充说明 (shapes, ranges), 约束说明,
 *                      返回值与错误码, Kernel 实现 (skip rules, fp32 math).
 * and around them: the batching from a ScheduleContext, its full-tail option,
 * the routing-map permute that produces the unpermute's input, and
 * MoeUpdateExpert ("MoeUpdateExpert"), declared further down.
 *
 * Conventions shared by every entry point
 *  - Pointers named as device pointers must point to device memory of the
 *    current CUDA device; pointers named host pointers to host memory.
 *  - The caller owns and frees every buffer, including the workspace. The
 *    library allocates no device memory and keeps no per-call state, with two
 *    exceptions, both created on first use and kept until exit:
 *    (1) the not-padded moe_unpermute keeps, per device and per caller
 *    `stream` (up to 64 caller streams per device), one auxiliary stream and
 *    two events: its sort of sortedIndices runs there, forked from and joined
 *    back into `stream`. Calls on different caller streams never share an
 *    auxiliary stream, so their sorts overlap and a stream capture on one
 *    caller stream does not reach calls on another. Past 64 caller streams
 *    on a device, the sort runs in `stream` itself.
 *    (2) ffnwb_batching_noalloc's fixed scratch array (see there).
 *    Both belong to the device's context: do not use the library across a
 *    cudaDeviceReset.
 *  - Execute calls are asynchronous on `stream` (a cudaStream_t; NULL = the
 *    legacy default stream). Outputs are valid once the caller synchronises
 *    the stream. Nothing is read back to the host.
 *  - Argument errors are detected on the host before anything is enqueued;
 *    the call then returns the error and enqueues nothing. Errors that the
 *    CUDA runtime reports at launch return MR_ERR_CUDA.
 *  - Outputs must not alias inputs or each other.
 *  - Results are deterministic: identical inputs give identical bits.
 *  - Execute calls can be captured into a CUDA graph (stream capture): they
 *    only enqueue kernels (the not-padded moe_unpermute's maskedSelect and
 *    the batching's one-launch sort of up to 32768 slots are cooperative
 *    launches, whose grids never exceed the blocks the device can hold at
 *    once), memsets and event records/waits on `stream` and its auxiliary
 *    stream, which joins back. Make one call of each kind on each caller
 *    stream outside any capture first (it creates that stream's auxiliary
 *    stream and caches device queries), and capture ffnwb_batching_noalloc
 *    only after its first call on the device.
 */
#ifndef MOE_REORDER_H
#define MOE_REORDER_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t mr_status;

/* Status codes. The first three carry the numeric values of the pages'
 * aclnnStatus codes ("aclnnFfnWorkerBatching" 返回值 table;
 * "MoeTokenUnpermuteWithRoutingMap 算子全解析" 返回值与错误码). */
#define MR_OK                 0
#define MR_ERR_PARAM_NULLPTR  161001 /* a required pointer is NULL */
#define MR_ERR_PARAM_INVALID  161002 /* dtype / shape / range out of the supported set */
#define MR_ERR_INNER          561103 /* topK_num > 512, or a probs shape out of range */
#define MR_ERR_CUDA           561001 /* the CUDA runtime reported an error */
#define MR_ERR_WORKSPACE      561002 /* workspaceSize smaller than required */
#define MR_ERR_UNSUPPORTED    561003 /* a valid mode this library does not implement */

/* Element types (tokenDtype / probsDtype). 0..2 are the batching page's
 * tokenDtype values; 3 is FP32 (allowed for the unpermute tensors). */
#define MR_DTYPE_F16   0
#define MR_DTYPE_BF16  1
#define MR_DTYPE_INT8  2 /* int8 rows with an fp32 dynamic scale */
#define MR_DTYPE_F32   3
#define MR_DTYPE_INT32 4 /* expert ids of moe_update_expert */
#define MR_DTYPE_INT64 5

/* Sentinel-free limits from the pages' constraint tables. */
#define MR_MAX_EXPERT_NUM 8192 /* expertNum in (0, 8192] */
#define MR_MAX_A          1024 /* A in (0, 1024] */
#define MR_MAX_TOPK1      64   /* topK+1 in (0, 64] */
#define MR_MAX_TOPK_NUM   512  /* unpermute topK_num <= 512 */
#define MR_MAX_UPDATE_BS      512  /* moe_update_expert: BS in (0, 512] */
#define MR_MAX_UPDATE_K       16   /* K in (0, 16], K <= moeExpertNum */
#define MR_MAX_UPDATE_EXPERTS 1024 /* moeExpertNum in (0, 1024] */

/* ------------------------------------------------------------------------ */
/* FFN-worker batching                                                      */
/* ------------------------------------------------------------------------ */

/*
 * ffnwb_batching_get_workspace_size
 *   "aclnnFfnWorkerBatching", 参数说明 (first-stage call) and 约束说明.
 *   Validates the attributes and returns, in *workspaceSize (host pointer),
 *   the bytes of device workspace ffnwb_batching needs.
 *
 *   expertNum    experts on this device over all layers, in (0, 8192].
 *   maxOutShape  host pointer to 4 int64: {A, BS, topK+1, H}; A in (0,1024],
 *                BS > 0, topK+1 in (0,64], H > 0. Y = A*BS*(topK+1) must be
 *                below 2^31.
 *   tokenDtype   MR_DTYPE_F16, MR_DTYPE_BF16 or MR_DTYPE_INT8.
 *   needSchedule 0 (batching only). 1 (scan the ScheduleContext first) needs
 *                the context's flags, which flat arrays do not have:
 *                MR_ERR_UNSUPPORTED here; ffnwb_batching_context
 *                implements it.
 *   layerNum     in [0, expertNum]; expertNum must be a multiple of
 *                max(layerNum, 1).
 *   Returns MR_OK, MR_ERR_PARAM_NULLPTR (maxOutShape or workspaceSize NULL),
 *   MR_ERR_PARAM_INVALID or MR_ERR_UNSUPPORTED.
 */
mr_status ffnwb_batching_get_workspace_size(int64_t expertNum, const int64_t* maxOutShape,
                                            int64_t tokenDtype, int64_t needSchedule,
                                            int64_t layerNum, uint64_t* workspaceSize);

/*
 * ffnwb_batching
 *   "aclnnFfnWorkerBatching", 功能说明 steps 2-4 and 计算公式:
 *     gather_idx, _ = sort(expert_ids_in)        (masked slots keyed last)
 *     y[i] = token_data[gather_idx[i]]           (+ dynamic scale, INT8)
 *     group_list[e] = [expert_id_e, expert_token_num_e]
 *     actual_token_num = sum_e expert_token_num_e
 *   The page's ScheduleContext is replaced by flat arrays of the Y slots
 *   (ffnwb_batching_context takes the context itself).
 *
 *   Inputs (device pointers unless noted; Y = A*BS*(topK+1) slots):
 *   expertIds       int32 [Y]: local expert id of each slot. A slot is masked
 *                   when its id is outside [0, E_l), E_l = expertNum /
 *                   max(layerNum,1) (e.g. INT32_MAX).
 *   layerId         the layer of every slot of this call, in
 *                   [0, max(layerNum,1)). Slot key = layerId*E_l + id.
 *   tokenData       Y rows, row s at tokenData + s*tokenRowStride bytes.
 *                   FP16/BF16: H values. INT8: H int8 values, and (when
 *                   scales is NULL) the fp32 scale in the 4 bytes right
 *                   after them.
 *   tokenRowStride  bytes between rows; >= H*elem (INT8 interleaved: >= H+4).
 *   scales          INT8 only, nullable: fp32 scale of slot s at
 *                   scales + s*scaleStride bytes.
 *   scaleStride     bytes between scales (ignored when scales is NULL).
 *   sessionIdsIn,
 *   microBatchIdsIn int32 [Y]: session / micro-batch id of each slot.
 *   tokenIdsIn      int32 [Y], nullable: token id of each slot; NULL means
 *                   the slot index.
 *   expertNum, maxOutShape (host), tokenDtype, needSchedule, layerNum:
 *                   as in ffnwb_batching_get_workspace_size.
 *   Outputs (device pointers; rows are in stable sort order of the key):
 *   y               [Y, H] of tokenDtype, dense rows. Rows i < U are written
 *                   (U = unmasked slots); rows i >= U are left untouched.
 *   groupList       int64 [expertNum, 2]: row r = [key, count] of the r-th
 *                   distinct present key in ascending order; remaining rows
 *                   [0, 0].
 *   sessionIds, microBatchIds, tokenIds, expertOffsets
 *                   int32 [Y]: ids of the slot in row i, and i minus the first
 *                   row of its key; -1 for rows i >= U.
 *   dynamicScale    float [Y]: INT8 only (must be NULL otherwise); rows i < U.
 *   actualTokenNum  int64 [1]: U.
 *   sortedIndicesOut int32 [Y], nullable: row of slot s in y, -1 if masked --
 *                   the sortedIndices of the unpermute's non-padded layout.
 *   workspace       device memory of at least the size the first stage
 *                   returned for the same attributes.
 *   stream          cudaStream_t.
 *   Returns MR_OK, MR_ERR_PARAM_NULLPTR, MR_ERR_PARAM_INVALID,
 *   MR_ERR_UNSUPPORTED, MR_ERR_WORKSPACE or MR_ERR_CUDA.
 */
mr_status ffnwb_batching(const int32_t* expertIds, int32_t layerId, const void* tokenData,
                         int64_t tokenRowStride, const void* scales, int64_t scaleStride,
                         const int32_t* sessionIdsIn, const int32_t* microBatchIdsIn,
                         const int32_t* tokenIdsIn, int64_t expertNum, const int64_t* maxOutShape,
                         int64_t tokenDtype, int64_t needSchedule, int64_t layerNum, void* y,
                         int64_t* groupList, int32_t* sessionIds, int32_t* microBatchIds,
                         int32_t* tokenIds, int32_t* expertOffsets, float* dynamicScale,
                         int64_t* actualTokenNum, int32_t* sortedIndicesOut, void* workspace,
                         uint64_t workspaceSize, void* stream);

/*
 * ffnwb_batching_ex
 *   ffnwb_batching with option flags (before the workspace arguments).
 *   MR_BATCHING_FULL_TAIL: apply 计算公式's y[i] = token_data[gather_idx[i]]
 *   and step 3's id lookup to the masked rows too: rows i >= U get the row,
 *   the INT8 scale and the session / micro-batch / token ids of the masked
 *   slot they hold (masked slots in ascending slot order); expertOffsets stays
 *   -1 there (a masked row is in no expert group). groupList, actualTokenNum
 *   and sortedIndicesOut are those of ffnwb_batching. Costs (Y - U) more row
 *   copies. Other flag bits: MR_ERR_PARAM_INVALID. ffnwb_batching is this call
 *   with flags 0; the workspace size is the same.
 */
#define MR_BATCHING_FULL_TAIL 1u
mr_status ffnwb_batching_ex(const int32_t* expertIds, int32_t layerId, const void* tokenData,
                            int64_t tokenRowStride, const void* scales, int64_t scaleStride,
                            const int32_t* sessionIdsIn, const int32_t* microBatchIdsIn,
                            const int32_t* tokenIdsIn, int64_t expertNum,
                            const int64_t* maxOutShape, int64_t tokenDtype, int64_t needSchedule,
                            int64_t layerNum, void* y, int64_t* groupList, int32_t* sessionIds,
                            int32_t* microBatchIds, int32_t* tokenIds, int32_t* expertOffsets,
                            float* dynamicScale, int64_t* actualTokenNum,
                            int32_t* sortedIndicesOut, uint32_t flags, void* workspace,
                            uint64_t workspaceSize, void* stream);

/*
 * ffnwb_batching_context_get_workspace_size / ffnwb_batching_context
 *   "aclnnFfnWorkerBatching", 功能说明 step 1 (read the FFN side's data area),
 *   参数说明 (scheduleContext, needSchedule) and the ScheduleContext /
 *   FfnDataDesc structs of 调用示例: the batching of ffnwb_batching with the
 *   page's own input, a packed 1024-byte ScheduleContext in device memory.
 *
 *   scheduleContext  device pointer, 8-byte aligned, 1024 bytes: CommonArea at
 *                    0 (u32 session_num, micro_batch_num, micro_batch_size,
 *                    selected_expert_num, expert_num = experts per layer),
 *                    FfnArea at 384 (u64 token_info_buf, token_info_buf_size,
 *                    token_data_buf, token_data_buf_size; device addresses).
 *                    token_info_buf holds one block per (session, micro-batch),
 *                    sessions outer: i32 flag, i32 layer_id, then
 *                    micro_batch_size * selected_expert_num i32 expert ids.
 *                    token_data_buf holds one row per slot in the same order:
 *                    H values (FP16/BF16) or H int8 values and their fp32
 *                    scale (INT8, stride H + 4), at any alignment (FP16/BF16
 *                    rows of whole 16-byte vectors at a 16-byte aligned
 *                    address copy fastest; the kernel checks the address).
 *   Slot g of block b: session id b / micro_batch_num, micro-batch id
 *   b % micro_batch_num, token id g, key = layer_id(b) * E_l + id (masked if
 *   the id or the block's layer is out of range).
 *   needSchedule     0: use every block. 1: a block takes part only once its
 *                    flag reads 1; the kernel waits for each flag until
 *                    waitTimeoutUs (at most 60 s) after it starts, and masks
 *                    the blocks still not ready.
 *   scheduleStatus   int32 [1], nullable device output: the number of blocks
 *                    that were not ready, or -1 if the context does not fit
 *                    (a count is 0, the slots exceed Y = A*BS*(topK+1) of
 *                    maxOutShape, expert_num != E_l, or a buffer is NULL,
 *                    misaligned or too small); then every slot is masked.
 *   The other arguments and the outputs are those of ffnwb_batching (outputs
 *   sized for Y rows; rows past the context's slots are part of the masked
 *   tail). The context is read on the device; nothing is synchronised.
 *   Returns the codes of ffnwb_batching.
 */
mr_status ffnwb_batching_context_get_workspace_size(int64_t expertNum, const int64_t* maxOutShape,
                                                    int64_t tokenDtype, int64_t needSchedule,
                                                    int64_t layerNum, uint64_t* workspaceSize);
mr_status ffnwb_batching_context(const void* scheduleContext, int64_t expertNum,
                                 const int64_t* maxOutShape, int64_t tokenDtype,
                                 int64_t needSchedule, int64_t layerNum, int64_t waitTimeoutUs,
                                 void* y, int64_t* groupList, int32_t* sessionIds,
                                 int32_t* microBatchIds, int32_t* tokenIds, int32_t* expertOffsets,
                                 float* dynamicScale, int64_t* actualTokenNum,
                                 int32_t* scheduleStatus, void* workspace, uint64_t workspaceSize,
                                 void* stream);
/*
 * ffnwb_batching_context_ex
 *   ffnwb_batching_context with option flags (before the workspace
 *   arguments); MR_BATCHING_FULL_TAIL as for ffnwb_batching_ex, for the slots
 *   the context holds: rows for slots past the context's (or every row of a
 *   context that does not fit) stay untouched, ids -1. ffnwb_batching_context
 *   is this call with flags 0.
 */
mr_status ffnwb_batching_context_ex(const void* scheduleContext, int64_t expertNum,
                                    const int64_t* maxOutShape, int64_t tokenDtype,
                                    int64_t needSchedule, int64_t layerNum, int64_t waitTimeoutUs,
                                    void* y, int64_t* groupList, int32_t* sessionIds,
                                    int32_t* microBatchIds, int32_t* tokenIds,
                                    int32_t* expertOffsets, float* dynamicScale,
                                    int64_t* actualTokenNum, int32_t* scheduleStatus,
                                    uint32_t flags, void* workspace, uint64_t workspaceSize,
                                    void* stream);

/*
 * ffnwb_batching_noalloc -- the batching for callers that cannot allocate.
 *   No counterpart on the pages: the pages' two-stage calls always take a
 *   caller-allocated workspace. Some callers cannot allocate device memory
 *   when they call, e.g. a plugin inside an engine that reserved all device
 *   memory at start-up, or a latency-critical loop that cannot afford
 *   cudaMalloc's implicit synchronisation. This entry point computes exactly
 *   what ffnwb_batching computes, with the same arguments minus the workspace,
 *   and allocates nothing: its scratch is a fixed array of
 *   MR_NOALLOC_SCRATCH_BYTES compiled into the library, which a GPU holds
 *   from the moment the library's code is loaded there until the process
 *   exits. Under CUDA's default lazy module loading that is the first call
 *   on the device, which may therefore allocate: make one call per device
 *   during start-up (before reserving the device's memory), or set
 *   CUDA_MODULE_LOADING=EAGER. Later calls allocate nothing.
 *   - Calls that need more scratch than the array holds return
 *     MR_ERR_WORKSPACE (4 MiB covers, e.g., Y = 147456 slots with
 *     expertNum = 8192, or Y = 262144 slots with expertNum = 1024).
 *   - All calls on a device share the array: calls whose work overlaps on the
 *     GPU (e.g. two streams at once) race; order them.
 *   - The first call on a device looks up the array's address on that device
 *     and caches it; make that first call before any stream capture.
 *   Returns the codes of ffnwb_batching.
 */
#define MR_NOALLOC_SCRATCH_BYTES (4u * 1024u * 1024u)
mr_status ffnwb_batching_noalloc(const int32_t* expertIds, int32_t layerId, const void* tokenData,
                                 int64_t tokenRowStride, const void* scales, int64_t scaleStride,
                                 const int32_t* sessionIdsIn, const int32_t* microBatchIdsIn,
                                 const int32_t* tokenIdsIn, int64_t expertNum,
                                 const int64_t* maxOutShape, int64_t tokenDtype,
                                 int64_t needSchedule, int64_t layerNum, void* y,
                                 int64_t* groupList, int32_t* sessionIds, int32_t* microBatchIds,
                                 int32_t* tokenIds, int32_t* expertOffsets, float* dynamicScale,
                                 int64_t* actualTokenNum, int32_t* sortedIndicesOut, void* stream);

/* ------------------------------------------------------------------------ */
/* Routing-map unpermute                                                    */
/* ------------------------------------------------------------------------ */

/*
 * moe_unpermute_get_workspace_size
 *   "MoeTokenUnpermuteWithRoutingMap 算子全解析", 调用说明 (first stage),
 *   功能说明与计算公式 (derived sizes), 约束说明, 返回值与错误码.
 *
 *   permutedRows      rows of permutedTokens (size(0)).
 *   hidden            H = permutedTokens.size(1) > 0.
 *   tokenDtype        MR_DTYPE_F16, MR_DTYPE_BF16 or MR_DTYPE_F32.
 *   numSortedIndices  n = len(sortedIndices).
 *   hasProbs          1 if probs and routingMap are given, else 0.
 *   probsDtype        tokenDtype or MR_DTYPE_F32 (ignored without probs).
 *   numTokens         T = probs.size(0) = routingMap.size(0) (with probs).
 *   numExperts        probs.size(1) (with probs).
 *   paddedMode        0 or 1.
 *   restoreShape      host pointer, nullable: {T, H} of the output. Required
 *                     without probs (it gives T); must agree with numTokens
 *                     and hidden otherwise.
 *   Derived: topK_num = permutedRows / T. Not padded: n == T*topK_num.
 *   Padded: n == permutedRows, capacity = n / numExperts (with probs n must be
 *   a multiple of numExperts).
 *   Returns MR_OK, MR_ERR_PARAM_NULLPTR, MR_ERR_PARAM_INVALID or MR_ERR_INNER
 *   (topK_num > 512, or the probs shape out of range).
 */
mr_status moe_unpermute_get_workspace_size(int64_t permutedRows, int64_t hidden,
                                           int32_t tokenDtype, int64_t numSortedIndices,
                                           int32_t hasProbs, int32_t probsDtype,
                                           int64_t numTokens, int64_t numExperts,
                                           int32_t paddedMode, const int64_t* restoreShape,
                                           uint64_t* workspaceSize);

/*
 * moe_unpermute
 *   "MoeTokenUnpermuteWithRoutingMap 算子全解析", 功能说明与计算公式:
 *   (1) probs, padded:     permuteProbs[i] = probs[sortedIndices[i], i // capacity];
 *                          permuteTokenId, outIndex = sortedIndices.sort();
 *                          out[permuteTokenId[i]] += permuted[outIndex[i]] * permuteProbs[outIndex[i]]
 *   (2) probs, not padded: permuteProbs = probs.T.maskedSelect(routingMap.T);
 *                          out[i // topK_num] += permuted[sortedIndices[i]] * permuteProbs[i]
 *   (3), (4): the same without probs.
 *   A term is skipped unless its index is valid (not padded:
 *   0 <= idx < permutedRows; padded: 0 <= token < T) and, with probs, its
 *   prob is nonzero. Terms are cast to fp32, multiplied by the fp32 prob,
 *   rounded, and added in fp32 in ascending slot (not padded) or row
 *   (padded) order; the sum is cast back with round-to-nearest-even.
 *   Tokens without a term get 0.
 *
 *   Inputs (device pointers):
 *   permutedTokens  [permutedRows, H] of tokenDtype.
 *   sortedIndices   int32 [n].
 *   routingMap      int8/bool [T, numExperts], nullable; NULL iff probs NULL.
 *   probs           [T, numExperts] of probsDtype, nullable.
 *   (shape arguments as in moe_unpermute_get_workspace_size)
 *   Outputs (device pointers):
 *   unpermutedTokens [T, H] of tokenDtype.
 *   outIndex         int32 [n]: positions of the stable ascending sort of
 *                    sortedIndices. Not padded: invalid entries first.
 *                    Padded: invalid entries last.
 *   permuteTokenId   int32 [n]: not padded: outIndex // topK_num; padded: the
 *                    sorted values (sortedIndices[outIndex[i]]).
 *   permuteProbs     [n] of probsDtype, required with probs, ignored without:
 *                    not padded: the maskedSelect values, truncated to n,
 *                    then zeros; padded: the lookup above, 0 where the index
 *                    is invalid.
 *   workspace, workspaceSize, stream: as for ffnwb_batching.
 *   Returns MR_OK, MR_ERR_PARAM_NULLPTR, MR_ERR_PARAM_INVALID, MR_ERR_INNER,
 *   MR_ERR_WORKSPACE or MR_ERR_CUDA.
 */
mr_status moe_unpermute(const void* permutedTokens, const int32_t* sortedIndices,
                        const int8_t* routingMap, const void* probs, int64_t permutedRows,
                        int64_t hidden, int32_t tokenDtype, int64_t numSortedIndices,
                        int32_t probsDtype, int64_t numTokens, int64_t numExperts,
                        int32_t paddedMode, const int64_t* restoreShape, void* unpermutedTokens,
                        int32_t* outIndex, int32_t* permuteTokenId, void* permuteProbs,
                        void* workspace, uint64_t workspaceSize, void* stream);

/*
 * moe_permute_get_workspace_size / moe_permute
 *   "MoeTokenUnpermuteWithRoutingMap 算子全解析", 算子定位: the permute step
 *   that precedes the unpermute rearranges the tokens by routingMap into an
 *   expert-grouped compact layout (permutedTokens), so each expert reads its
 *   tokens contiguously. The page names this step without its formulas; the
 *   layouts below are the ones moe_unpermute takes.
 *
 *   tokens          [numTokens, hidden] of tokenDtype (F16, BF16 or F32).
 *   routingMap      int8/bool [numTokens, numExperts]; numExperts in [1, 8192].
 *   paddedMode 0    topK in [1, 512] slots per token (561103 above 512).
 *                   permutedTokens [numTokens*topK, hidden]: the routed
 *                   (token, expert) pairs in expert-major order (expert, then
 *                   token ascending) -- the order of probs.T.maskedSelect(
 *                   routingMap.T); rows past the pairs are not written.
 *                   sortedIndices int32 [numTokens*topK]: slot t*topK + j =
 *                   row of t's j-th routed expert (ascending id), -1 for j at
 *                   or past its count and for a pair whose row would be past
 *                   numTokens*topK.
 *   paddedMode 1    capacity >= 1. permutedTokens [numExperts*capacity,
 *                   hidden]: expert e keeps its first `capacity` routed tokens
 *                   (ascending token id) in rows e*capacity + r; the other
 *                   rows are zero. sortedIndices int32 [numExperts*capacity]:
 *                   the row's token id, -1 for a padding row.
 *   permutedRowsOut int32 [1], nullable: rows written from tokens (not
 *                   padded: min(pairs, numTokens*topK); padded: rows kept).
 *   Returns MR_OK, MR_ERR_PARAM_NULLPTR, MR_ERR_PARAM_INVALID, MR_ERR_INNER,
 *   MR_ERR_WORKSPACE or MR_ERR_CUDA.
 */
mr_status moe_permute_get_workspace_size(int64_t numTokens, int64_t hidden, int32_t tokenDtype,
                                         int64_t numExperts, int64_t topK, int32_t paddedMode,
                                         int64_t capacity, uint64_t* workspaceSize);
mr_status moe_permute(const void* tokens, const int8_t* routingMap, int64_t numTokens,
                      int64_t hidden, int32_t tokenDtype, int64_t numExperts, int64_t topK,
                      int32_t paddedMode, int64_t capacity, void* permutedTokens,
                      int32_t* sortedIndices, int32_t* permutedRowsOut, void* workspace,
                      uint64_t workspaceSize, void* stream);

/*
 * moe_update_expert
 *   "MoeUpdateExpert", 功能说明 and 参数说明: maps each token's top-K logical
 *   expert ids to physical expert instances through the EPLB table (load
 *   balancing), and prunes a token's experts whose scale is below a threshold.
 *   The page gives no formula for the choice of instance; this library reads
 *   "by rank" and "by token" as
 *     balancedExpertIds[b,k] = eplbTable[e, 1 + c], e = expertIds[b,k],
 *     count = eplbTable[e, 0], c = localRankId mod count (balanceMode 0) or
 *     c = b mod count (balanceMode 1);
 *   -1 when e is outside [0, moeExpertNum) or count outside [1, F - 1] (no
 *   read leaves the table). With scales and threshold:
 *     balancedActiveMask[b,k] = activeMask[b] && !(f32(scale[b,k]) < threshold[k])
 *   (equal is kept; activeMask NULL means every token is active).
 *
 *   Inputs (device pointers):
 *   expertIds          [BS, K] of idDtype (MR_DTYPE_INT32 or MR_DTYPE_INT64).
 *   eplbTable          int32 [moeExpertNum, F]: column 0 the instance count,
 *                      columns 1..count the instance ids.
 *   expertScales       [BS, K] of scalesDtype (F16, BF16, F32), nullable;
 *                      NULL iff pruningThreshold is NULL.
 *   pruningThreshold   float32 [K], nullable.
 *   activeMask         bool (one byte, nonzero = true) [BS], nullable; needs
 *                      expertScales. The page asks that the trues come first;
 *                      the result does not depend on it.
 *   BS in (0, 512]; K in (0, 16], K <= moeExpertNum; moeExpertNum in
 *   (0, 1024]; balanceMode 0: worldSize in [2, 768], localRankId in
 *   [0, worldSize); balanceMode 1: worldSize in [1, 1024], localRankId unused;
 *   F in [2, worldSize + 1].
 *   strides            host array of 12 int64 element strides, nullable (NULL:
 *                      contiguous): expertIds (b, k), eplbTable (e, f),
 *                      expertScales (b, k), pruningThreshold (k), activeMask
 *                      (b), balancedExpertIds (b, k), balancedActiveMask (b, k).
 *                      Input strides >= 0 (0 broadcasts), output strides >= 1.
 *                      Read during the call only.
 *   Outputs (device pointers):
 *   balancedExpertIds  [BS, K] of idDtype.
 *   balancedActiveMask bool [BS, K]; required with expertScales, not written
 *                      without.
 *   stream             cudaStream_t (NULL: the legacy default stream). No
 *                      workspace is needed.
 *   Returns MR_OK, MR_ERR_PARAM_NULLPTR, MR_ERR_PARAM_INVALID or MR_ERR_CUDA.
 */
mr_status moe_update_expert(const void* expertIds, int32_t idDtype, const int32_t* eplbTable,
                            const void* expertScales, int32_t scalesDtype,
                            const float* pruningThreshold, const uint8_t* activeMask, int64_t BS,
                            int64_t K, int64_t moeExpertNum, int64_t F, int64_t localRankId,
                            int64_t worldSize, int64_t balanceMode, const int64_t* strides,
                            void* balancedExpertIds, uint8_t* balancedActiveMask, void* stream);

/* ------------------------------------------------------------------------ */
/* Utilities (no counterpart on the pages)                                  */
/* ------------------------------------------------------------------------ */

/* Short English text of a status code (static storage). */
const char* mr_status_string(mr_status status);

/* Library version, major*10000 + minor*100 + patch. */
int32_t mr_version(void);

/*
 * mr_profile_set_events -- timing aid for benchmarks.
 *   events: host array of `count` cudaEvent_t handles (count even, <= 16), or
 *   NULL / 0 to switch timing off. While set, the calling thread's execute
 *   calls record events[2p] before and events[2p+1] after phase p on their
 *   stream, phases being: 0 batching index build, 1 batching row gather,
 *   2 unpermute probs work (maskedSelect or the padded lookup; padded: also
 *   the sort), 3 unpermute gather-reduce, 4 the not-padded sort, which runs
 *   on the caller stream's auxiliary stream (its events are recorded there).
 *   Phases beyond `count/2` are not recorded.
 *   The setting is per host thread. Returns MR_OK or MR_ERR_PARAM_INVALID.
 */
mr_status mr_profile_set_events(void* const* events, int32_t count);

/*
 * mr_checked_errors -- the bounds checks of a checked build.
 *   No counterpart on the pages; its nearest relative is the unpermute
 *   kernel's IsValidInputIndex guard ("MoeTokenUnpermuteWithRoutingMap
 *   算子全解析", Kernel 实现), which skips a slot whose index is out of range.
 *   A library built with -DMR_CHECKED range-checks every gather index, row
 *   offset, CSR row pointer and scatter destination that a kernel derives
 *   from data (an input, a workspace word or another kernel's output); an
 *   access that fails its check is skipped and counted in a device error
 *   word. On valid inputs the count stays 0 and the outputs are those of the
 *   regular build. This call synchronises with the device, writes the number
 *   of failed checks since the last reset to *failures (host pointer) and
 *   the site number of the first one to *firstSite (host pointer, may be
 *   NULL), and with reset != 0 clears the words.
 *   Returns MR_OK, MR_ERR_PARAM_NULLPTR (failures NULL), MR_ERR_CUDA, or
 *   MR_ERR_UNSUPPORTED in a regular build (which has no checks; it writes 0).
 */
mr_status mr_checked_errors(uint32_t* failures, uint32_t* firstSite, int32_t reset);

#ifdef __cplusplus
}
#endif

#endif /* MOE_REORDER_H */
