"""GB300-native (sm_103a) shifted-schedule sharded attention.

The hot path of Mercury's shifted asynchronous schedule (SOSP 2025) on one
GPU: R virtual ranks, rank i consuming KV shard order[i][j] at step j, a
tcgen05/TMEM/TMA flash-attention forward "patch", and a log-sum-exp merge of
per-step partials.  The compute entry points live in ``mercury`` (a ctypes
binding of the in-tree libmercury_attn.so); importing them fails loudly when
the library has not been built.  ``inputs`` and ``workloads`` hold the seeded
synthetic inputs and workload shapes.
"""

__all__ = ["mercury_plan_shift", "mercury_attn_sharded", "mercury_attn_partial",
           "mercury_lse_merge", "mercury_sync_status", "MercuryError"]


def __getattr__(name):
    if name in __all__:
        from . import mercury
        return getattr(mercury, name)
    raise AttributeError(name)
