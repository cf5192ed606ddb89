"""Plain, slow, fp64 CPU oracle for selected-block attention.

THIS PACKAGE IS TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()``
and ``bench.py`` (its ``cpu_baseline`` leg and ``--impl reference`` arm) may
import it. The product package ``selected_block_attention_gb300`` never imports
it, and it imports nothing from the product package: the two share no code.

Every function works in float64 on numpy arrays and follows the passage of the
source documentation pages named in its docstring:

* ``nsa_select_attention``     -- ejkernel.modules.operations.native_sparse_attention
  (operation API page), ``NativeSparseAttention.run`` / ``native_sparse_attention``.
* ``sparse_mask_bounds``       -- ejkernel.kernels._triton.blocksparse_attention._mask
  (module source page), ``_compute_sparse_mask`` + ``define_sparse_mask_fn``.
* ``blocksparse_attention``    -- same page, module docstring and ``SparseMask``
  docstring (attention restricted to the [lower, upper) block range).
* ``ragged_decode_attention``  -- ejkernel.kernels._xla.ragged_decode_attention._xla_impl_fwd
  (API page), ``inner_decode_xla`` / ``create_attention_mask`` /
  ``apply_logits_soft_cap`` / ``apply_attention_sinks_block``.
* ``ragged_flash_attention``   -- same page, ``ragged_flash_attention_xla`` (Q queries
  per row, the last Q tokens of its range).
* ``nsa_select_attention_backward`` -- gradients (dq, dk, dv) of the selection
  forward, the softmax backward over the same explicit key sets.

Every function is pinned by ``tests/test_oracle_*.py`` against closed forms,
library routines (torch SDPA in float64), brute force on tiny inputs and the
worked example printed on the mask page.
"""

from .nsa import nsa_select_attention, selected_key_set
from .sparse_mask import sparse_mask_bounds
from .blocksparse import blocksparse_attention
from .ragged_decode import ragged_decode_attention
from .ragged_attention import ragged_flash_attention
from .nsa_backward import nsa_select_attention_backward

__all__ = [
    "nsa_select_attention",
    "selected_key_set",
    "sparse_mask_bounds",
    "blocksparse_attention",
    "ragged_decode_attention",
    "ragged_flash_attention",
    "nsa_select_attention_backward",
]
