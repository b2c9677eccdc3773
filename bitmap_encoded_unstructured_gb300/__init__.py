"""bitmap_encoded_unstructured_gb300: bitmap-encoded unstructured sparse matmul on GB300."""
