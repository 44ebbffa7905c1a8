"""GB300-native paged KV-cache decode attention (GQA / MQA / MHA and MLA)."""
