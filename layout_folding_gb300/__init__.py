"""layout_folding_gb300 -- placeholder, replaced by the binding module."""
