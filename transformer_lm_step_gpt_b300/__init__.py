"""B300-native GPT-2 training step (binding placeholder; filled in with the C ABI)."""
