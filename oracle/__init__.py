"""Float64 CPU oracle for the DeBERTa-v2/v3 disentangled-attention forward pass.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import this
package: only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
CPU-baseline / reference arm use it.  It shares no code with the CUDA path.
"""

from .df_oracle import (  # noqa: F401
    log_bucket,
    rel_index,
    attend_sequence,
    attend_padded,
    attend_packed,
    attend_rows,
    metric_flops,
)
from .pack import pack_info, pack_rows, unpack_rows  # noqa: F401,E402
from .linear import linear  # noqa: F401,E402
from .encoder import layer_norm, gelu, encoder_layer, encoder  # noqa: F401,E402
from .backward import (  # noqa: F401,E402
    backward_head,
    backward_rows,
    backward_keys,
    backward_sequence,
    backward_padded,
    backward_packed,
    backward_metric_flops,
)
