"""GB300-native path-conditioned draft-tree construction (libdtree + binding)."""
from .dtree import (  # noqa: F401
    DraftTreeBuilder,
    DtreeError,
    bf16_tensor,
    check_config,
    load_library,
    node_count,
    status_string,
    workspace_bytes,
)
