"""GB300-native split-KV sparse-MLA decode (placeholder; the binding lands with the C ABI)."""
