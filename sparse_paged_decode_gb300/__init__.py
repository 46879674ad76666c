"""sparse_paged_decode_gb300 -- decode-time sparse attention boundary for GB300.

Three stages behind a C ABI (``include/spd.h``), each a hand-written sm_103a
CUDA kernel:

  msa_block_score                 block-max score sheet over a paged index cache
  msa_select_topk                 top-k block ids per query row
  paged_sparse_decode_attention   paged GQA attention over the selected blocks
  paged_decode_attention          the same over every block (dense decode)
  msa_prefill_block_score         fused prefill score-to-selection per query block
  attention_sdpa                  dense (not paged) GQA attention, causal flag

The Python functions of the same names (in :mod:`.binding`) only marshal
torch tensors into the C ABI; every step runs in the CUDA library.  They
raise if the library has not been built: there is no CPU fallback.

``workloads`` draws the seeded synthetic inputs and imports nothing else.
"""

__all__ = [
    "msa_block_score",
    "msa_select_topk",
    "paged_sparse_decode_attention",
    "paged_decode_attention",
    "paged_sparse_decode_attention_noalloc",
    "attention_sdpa",
    "msa_prefill_block_score",
    "prefill_workspace_bytes",
    "decode_workspace_bytes",
    "launch_count",
    "set_attention_kernel",
    "set_kernel_policy",
    "workspace_status",
    "library_path",
]


def __getattr__(name):
    # the binding (and with it the CUDA library) loads on first use only, so
    # importing ``workloads`` pulls in nothing else
    if name in __all__:
        from . import binding

        return getattr(binding, name)
    raise AttributeError(name)
