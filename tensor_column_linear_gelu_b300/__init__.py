"""tensor_column_linear_gelu_b300 -- the Megatron-style tensor-parallel split of
a transformer layer's linear algebra (column-parallel linear + activation,
row-parallel linear + in-kernel shard sum + bias, FFN block, head-split
attention projections), every shard on one B300, in hand-written sm_103a CUDA
kernels behind a C ABI (include/tpla.h).

``tensor_column_linear_gelu_b300.tpla`` is the binding; importing it loads
libtpla.so and fails loudly if the library has not been built.
"""
_BINDING = ("tp_shard_shape", "tp_shard_weights", "column_parallel_linear",
            "row_parallel_linear", "tp_mlp_block", "tp_attn_proj", "tp_device_status",
            "tp_selftest_bounded_wait", "TplaError")


def __getattr__(name):
    if name in _BINDING:
        from . import tpla
        return getattr(tpla, name)
    raise AttributeError(name)
