"""GB300-native AdamW optimizer step (pure-bf16 Kahan and fp32-master mixed
modes) behind a small C ABI; see ``adamw_sm`` for the binding."""
