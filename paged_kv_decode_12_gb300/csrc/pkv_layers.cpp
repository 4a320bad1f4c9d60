// pkv_layers.cpp -- every layer of one decode step in one host call.
//
// The decode loop runs the model's layers in turn (samir-vllm README summary,
// "目前已完成的功能": one decode step appends the new token and attends over the
// pages of every layer).  pkv_decode_step_layers issues pkv_decode_step for layer
// 0 .. layers-1 in that order on one stream, so that a host loop makes one call per
// step instead of one per layer.  Host code only: the launches are pkv_decode_step's.
#include "pkv_internal.h"

// Layer l's per-layer arrays are the bases plus l strides (elements).  Layer 0 is
// validated and launched first, so an invalid argument launches nothing; the strides
// keep every later layer's pointers 16-byte aligned, so later layers pass the same
// checks.
extern "C" int pkv_decode_step_layers(const pkv_pool *pool, int layers, const uint16_t *k_new,
                                      const uint16_t *v_new, uint16_t *q, const int32_t *bt_dev, int max_blocks,
                                      const int32_t *seq_lens_dev, int B, const float *rope_table, int max_pos,
                                      float scale, int pages_per_chunk, void *workspace, size_t workspace_bytes,
                                      uint16_t *out, int32_t *dev_err_flag, void *cuda_stream, int options,
                                      int64_t kv_layer_stride, int64_t q_layer_stride, int64_t bt_layer_stride)
{
    if (layers < 1 || kv_layer_stride < 0 || q_layer_stride < 0 || bt_layer_stride < 0)
        return PKV_ERR_INVALID_ARG;
    if (layers > 1 && (((kv_layer_stride * 2) & 15) || ((q_layer_stride * 2) & 15)))
        return PKV_ERR_INVALID_ARG;  // every layer's BF16 rows stay 16-byte aligned
    for (int l = 0; l < layers; ++l) {
        const int st = pkv_decode_step(pool, k_new + l * kv_layer_stride, v_new + l * kv_layer_stride,
                                       q + l * q_layer_stride, bt_dev + l * bt_layer_stride, max_blocks, seq_lens_dev,
                                       B, rope_table, max_pos, scale, pages_per_chunk, workspace, workspace_bytes,
                                       out + l * q_layer_stride, dev_err_flag, cuda_stream, options);
        if (st != PKV_OK)
            return st;
    }
    return PKV_OK;
}
